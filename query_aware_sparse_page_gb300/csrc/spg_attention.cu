// Split-K flash-decoding over gathered KV pages, with the log-sum-exp merge
// of the splits done by the last CTA of each unit.
//
// Sources: SALS长序列推理优化, SFAA (QK^T, online softmax, P@V, rescale over
// the selected K/V; int8 K/V dequantised by their scales) and AICPU Tiling
// challenge 2 (a row split over several cores is merged by a reduction);
// Quest 完全拆解, 三段式 kernel (Approximate attention reads only the top-K
// pages); Day 10·2 (softmax renormalised over the selected blocks only).
//
// Grid = (splits, batch * kv-heads), sized to one wave, for a selection (the
// units' counts are alike).  The dense baseline plans its split by length
// (SALS AICPU Tiling: the work of a ragged batch divided by a cost model of
// each row's length): the grid is one wave of CTAs, and every CTA computes
// the same plan from seq_lens, unit u taking parts(u) = ceil(w_u N / T)
// consecutive CTAs (w_u its pages, T = sum of w_u, N = the CTAs less one per
// unit, so that the rounding still fits the wave; 1 <= parts(u) <= the
// split limit), then finds its own (unit, part) by a prefix over the units;
// the parts of a unit cover its pages in equal contiguous ranges.  A CTA owns
// a contiguous range of the unit's page list (selected ids, or every page for
// the dense baseline) and is warp-specialised:
//  * the producer warp resolves logical -> physical page ids 32 at a time
//    (one lane per page) and streams each page's K and V tiles ([S][d] of one
//    kv-head in the [P][Hkv][S][d] pools, plus the per-token fp16 scales for
//    int8) into a shared-memory ring of stages of up to 8 pages, one lane per
//    page: 2-D TMA tiles with 128-byte swizzle for the tensor-core consumers,
//    cp.async.bulk otherwise; one "full" mbarrier per stage carries the bytes;
//  * stage k belongs to consumer warp k % 4, which runs the flash-decoding
//    consumer over its pages (tensor cores for fp16/bf16 pages and for int8
//    pages of head_dim 128 with an fp16 query, CUDA cores otherwise) and
//    releases the stage on its "empty" mbarrier.
// Each of the G query rows of the kv-head group reuses every staged tile
// (GQA).  All waits are bounded; a wait that runs out records
// SPG_DEVERR_TIMEOUT and the CTA drains (again bounded) the copies it issued
// before it leaves.
//
// Partials per (batch, q-head, split): running max m (log2 domain, scale
// folded in), running sum l, unnormalised accumulator acc[d].  The last CTA
// of a unit to arrive (an atomic counter per unit in the workspace, reset by
// that CTA) merges the unit's splits and writes out and lse, so one launch
// does the whole attention.
#include <float.h>

#include "spg_attn_core.cuh"
#include "spg_internal.h"

namespace spg {
namespace {

constexpr int kRingBytesTarget = 64 * 1024;
constexpr int kStageBytesTarget = 16 * 1024;
constexpr int kMaxPagesPerStage = 8;

struct AttnArgs {
  CUtensorMap tmk, tmv;  // K / V pools as page tiles (tensor-core consumers)
  int whole_page;        // the maps are 3-D: one copy per page
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const __half* k_scale;
  const __half* v_scale;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* sel;      // nullptr -> dense
  const int32_t* sel_cnt;
  float* pm;
  float* pl;
  float* pacc;
  int32_t* counters;  // split arrivals per unit, zero between launches
  int planned;        // dense: (unit, part) from the length plan (grid = (CTAs, 1))
  int units, plan_n;  // units; N of the plan (CTAs less one per unit)
  int32_t* hook;      // test hook (workspace header): withhold the first stage of CTA (0, 0)
  float* out;
  float* lse;
  int32_t* err;
  int Hkv, S, MP, n_phys, n_sel, pages_per_split, stages, pages_per_stage;
  uint32_t stage_bytes, page_bytes;
  float scale_log2;
};

template <typename T, typename TQ, int D, int G>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32)
    k_attn(const __grid_constant__ AttnArgs a) {
  constexpr int CW = kConsumerWarps;
  // consumer: 1 = tensor cores on fp16/bf16 pages, 2 = tensor cores on int8
  // pages (D = 128, fp16 query), 0 = CUDA cores; 1 and 2 take TMA tiles
  constexpr int CONS = !is_i8<T>() ? 1 : ((D == 128 && std::is_same<TQ, __half>::value) ? 2 : 0);
  constexpr bool MMA = CONS != 0;
  using Consumer = std::conditional_t<
      CONS == 1, AttnMma<T, D, G>,
      std::conditional_t<CONS == 2, AttnMmaI8<G>, AttnConsumer<T, D, G, 1>>>;

  extern __shared__ __align__(128) uint8_t smem_raw[];
  // TMA tiles with 128-byte swizzle want 1024-byte aligned destinations
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = a.S;
  const int STAGES = a.stages, PPS = a.pages_per_stage;
  const uint32_t tile = static_cast<uint32_t>(S) * D * sizeof(T);
  const uint32_t scb = is_i8<T>() ? static_cast<uint32_t>(S) * 2 : 0u;
  const uint32_t sbytes = a.stage_bytes, pbytes = a.page_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(STAGES) * sbytes);
  uint64_t* empty = full + kMaxStages;
  int* s_np = reinterpret_cast<int*>(empty + kMaxStages);  // [stages] pages in stage
  int* s_nv = s_np + kMaxStages;                          // [stages][8] valid tokens
  __shared__ int s_last;
  __shared__ int s_plan[3];  // unit, part, parts of the unit

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = a.Hkv;
  int unit = blockIdx.y, split = blockIdx.x, n_parts = gridDim.x;
  int pages_per_split = a.pages_per_split;
  if (a.planned) {
    // the length plan (every CTA computes the same one) from seq_lens, which
    // a previous kernel may have written
    pdl_wait();
    if (warp == 0) {
      long long T = 0;
      const int B = a.units / Hkv;
      for (int bb = lane; bb < B; bb += 32) {
        const int Lb = a.seq_lens[bb];
        T += (Lb > 0 && Lb <= a.MP * a.S) ? (Lb + a.S - 1) / a.S : 0;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) T += __shfl_xor_sync(0xffffffffu, T, o);
      T *= Hkv;
      int found_u = -1, found_j = 0, found_n = 1;
      long long base = 0;
      for (int u0 = 0; u0 < a.units; u0 += 32) {
        const int u = u0 + lane;
        int parts = 0;
        if (u < a.units) {
          const int Lb = a.seq_lens[u / Hkv];
          const long long w = (Lb > 0 && Lb <= a.MP * a.S) ? (Lb + a.S - 1) / a.S : 0;
          parts = T > 0 ? static_cast<int>((w * a.plan_n + T - 1) / T) : 1;
          parts = max(1, min(kMaxSplits, parts));
        }
        int incl = parts;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const long long lo = base + incl - parts;
        if (u < a.units && blockIdx.x >= lo && blockIdx.x < lo + parts) {
          found_u = u;
          found_j = static_cast<int>(blockIdx.x - lo);
          found_n = parts;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      const unsigned hit = __ballot_sync(0xffffffffu, found_u >= 0);
      if (lane == 0) s_plan[0] = -1;
      __syncwarp();
      if (found_u >= 0 && (hit & ((1u << lane) - 1u)) == 0) {
        s_plan[0] = found_u;
        s_plan[1] = found_j;
        s_plan[2] = found_n;
      }
    }
    __syncthreads();
    if (s_plan[0] < 0) return;  // past the plan's last part: no work, nothing shared
    unit = s_plan[0];
    split = s_plan[1];
    n_parts = s_plan[2];
  }
  const int b = unit / Hkv, h = unit % Hkv;
  const int Hq = Hkv * G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_fence_init();
  }
  if constexpr (MMA) {
    if (threadIdx.x == CW * 32) {
      tma_prefetch_desc(&a.tmk);
      tma_prefetch_desc(&a.tmv);
    }
  }
  pdl_wait();  // sel / sel_cnt (and anything else) may come from the previous kernel

  int L = a.seq_lens[b];
  if (L < 0 || L > a.MP * S) {
    if (split == 0 && threadIdx.x == 0) record_error(a.err, SPG_DEVERR_SEQ_LEN);
    L = 0;
  }
  const int P = (L + S - 1) / S;
  int count = P;
  if (a.sel) {
    count = a.sel_cnt[unit];
    if (count < 0 || count > a.n_sel) {
      if (split == 0 && threadIdx.x == 0) record_error(a.err, SPG_DEVERR_SEL);
      count = max(0, min(count, a.n_sel));
    }
  }
  int s0, n_range;
  if (a.planned) {  // the part's share of the unit's pages
    s0 = static_cast<int>(static_cast<long long>(split) * count / n_parts);
    n_range = static_cast<int>(static_cast<long long>(split + 1) * count / n_parts) - s0;
  } else {
    s0 = split * pages_per_split;
    n_range = max(min(s0 + pages_per_split, count) - s0, 0);
  }
  const int n_st = (n_range + PPS - 1) / PPS;
  __syncthreads();

  Consumer cons;

  if (warp == CW) {
    // ---------------- producer: page ids, then one lane per page of a stage
    const T* kpool = static_cast<const T*>(a.k_pool);
    const T* vpool = static_cast<const T*>(a.v_pool);
    const uint64_t pol = policy_evict_first();
    bool ok = true;
    // test hook (spg_test_withhold_first_stage): CTA (0, 0) issues no copy
    // for its first stage and never completes it, so that the consumer's
    // bounded wait runs out with nothing in flight; one shot
    bool withhold = false;
    if (a.hook && split == 0 && unit == 0) {
      int hv = 0;
      if (lane == 0) hv = atomicExch(a.hook, 0);
      withhold = __shfl_sync(0xffffffffu, hv, 0) != 0;
    }
    for (int base = 0; base < n_range && ok; base += 32) {
      int ph = -1, nv = 0;
      const int j = base + lane;
      if (j < n_range) {
        const int idx = s0 + j;
        const int lp = a.sel ? a.sel[static_cast<size_t>(unit) * a.n_sel + idx] : idx;
        if (lp < 0 || lp >= P) {
          record_error(a.err, SPG_DEVERR_SEL);
        } else {
          ph = a.page_table[static_cast<size_t>(b) * a.MP + lp];
          if (ph < 0 || ph >= a.n_phys) {
            record_error(a.err, SPG_DEVERR_PAGE_ID);
            ph = -1;
          } else {
            nv = min(S, L - lp * S);
          }
        }
      }
      const int nb = min(32, n_range - base);
      for (int t0 = 0; t0 < nb && ok; t0 += PPS) {
        const int k = (base + t0) / PPS, stage = k % STAGES;
        bool lok = true;
        if (lane == 0 && k >= STAGES) lok = mbar_wait_bounded(&empty[stage], ((k / STAGES) - 1) & 1);
        if (!lok) record_error(a.err, SPG_DEVERR_TIMEOUT);
        ok = __shfl_sync(0xffffffffu, lok ? 1 : 0, 0) != 0;
        if (!ok) break;
        const int np = min(PPS, nb - t0);
        if (withhold && k == 0) continue;  // no copy, no arrival: the stage never completes
        if (lane >= t0 && lane < t0 + np) {
          const int i = lane - t0;
          uint8_t* dst = smem + static_cast<size_t>(stage) * sbytes + static_cast<size_t>(i) * pbytes;
          s_nv[stage * kMaxPagesPerStage + i] = ph >= 0 ? nv : 0;
          if (ph >= 0) {
            const size_t row = static_cast<size_t>(ph) * Hkv + h;
            mbar_expect_tx(&full[stage], 2 * tile + 2 * scb);
            if constexpr (MMA) {
              // swizzled tiles of [S rows][128 bytes] for K, then for V
              constexpr int NT = D * static_cast<int>(sizeof(T)) / 128, EPT = 128 / sizeof(T);
              const int y = static_cast<int>(row) * S;
              if (a.whole_page) {
                tma_load_3d(dst, &a.tmk, 0, y, 0, &full[stage], pol);
                tma_load_3d(dst + tile, &a.tmv, 0, y, 0, &full[stage], pol);
              } else {
#pragma unroll
                for (int hf = 0; hf < NT; ++hf) {
                  tma_load_2d(dst + hf * S * 128, &a.tmk, hf * EPT, y, &full[stage], pol);
                  tma_load_2d(dst + tile + hf * S * 128, &a.tmv, hf * EPT, y, &full[stage], pol);
                }
              }
            } else {
              bulk_g2s_hint(dst, kpool + row * S * D, tile, &full[stage], pol);
              bulk_g2s_hint(dst + tile, vpool + row * S * D, tile, &full[stage], pol);
            }
            if constexpr (is_i8<T>()) {
              bulk_g2s(dst + 2 * tile, a.k_scale + row * S, scb, &full[stage]);
              bulk_g2s(dst + 2 * tile + scb, a.v_scale + row * S, scb, &full[stage]);
            }
          }
        }
        if (lane == 0) s_np[stage] = np;
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);
      }
    }
    if (!ok && lane == 0) {
      // drain the copies still in flight before the CTA can leave (bounded
      // waits; uses that were never issued simply time out)
      for (int k = max(0, n_st - STAGES); k < n_st; ++k)
        mbar_wait_bounded(&full[k % STAGES], (k / STAGES) & 1);
    }
  } else {
    // ---------------- consumers: stage k belongs to warp k % CW
    cons.init(static_cast<const TQ*>(a.q) + (static_cast<size_t>(b) * Hq + h * G) * D,
              a.scale_log2, warp, lane);
    for (int k = warp; k < n_st; k += CW) {
      const int stage = k % STAGES;
      if (!mbar_wait_bounded(&full[stage], (k / STAGES) & 1)) {
        if (lane == 0) record_error(a.err, SPG_DEVERR_TIMEOUT);
        break;
      }
      const int np = s_np[stage];
      for (int i = 0; i < np; ++i) {
        const int nv = s_nv[stage * kMaxPagesPerStage + i];
        uint8_t* pg = smem + static_cast<size_t>(stage) * sbytes + static_cast<size_t>(i) * pbytes;
        if (nv > 0) {
          if constexpr (MMA)
            cons.consume(pg, S, nv, lane);
          else
            cons.consume(pg, S, nv);
        }
      }
      if constexpr (MMA) fence_proxy_async();  // zeroed slots before the next TMA write
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    cons.fold();
  }

  pdl_trigger();
  // merge the consumer warps of this CTA (reusing the ring), write the partial
  __syncthreads();
  float* s_m = reinterpret_cast<float*>(smem);  // [CW][G]
  float* s_l = s_m + CW * G;                     // [CW][G]
  float* s_acc = s_l + CW * G;                   // [CW][G][D]
  if (warp < CW) cons.store(s_m, s_l, s_acc, lane);
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D, c = idx % D;
    float M, Ls, A;
    lse_merge(s_m, s_l, s_acc, CW, G, D, g, c, M, Ls, A);
    const size_t row = static_cast<size_t>(b) * Hq + h * G + g;
    const size_t pidx = row * kMaxSplits + split;
    a.pacc[pidx * D + c] = A;
    if (c == 0) {
      a.pm[pidx] = M;
      a.pl[pidx] = Ls;
    }
  }

  // The last CTA of the unit to finish merges every split by log-sum-exp
  // (SALS AICPU Tiling, challenge 2: the reduction of a row split across
  // cores).  Writers publish their partials with a device-scope fence before
  // counting themselves in; no CTA ever waits for another.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(&a.counters[unit], 1);
    s_last = (prev == n_parts - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int n_split = n_parts;
  // weights of every split per row, in shared memory (reusing the ring)
  float* s_w = reinterpret_cast<float*>(smem);  // [G][n_split]
  float* s_M = s_w + G * kMaxSplits;            // [G]
  float* s_L = s_M + G;                         // [G]
  for (int g = warp; g < G; g += CW + 1) {
    const size_t row = static_cast<size_t>(b) * Hq + h * G + g;
    const float* pmr = a.pm + row * kMaxSplits;
    const float* plr = a.pl + row * kMaxSplits;
    float M = -INFINITY;
    for (int sp = lane; sp < n_split; sp += 32) M = fmaxf(M, __ldcg(pmr + sp));
    M = warp_max(M);
    float Ls = 0.f;
    for (int sp = lane; sp < n_split; sp += 32) {
      const float f = M == -INFINITY ? 0.f : exp2f(__ldcg(pmr + sp) - M);
      s_w[g * kMaxSplits + sp] = f;
      Ls = fmaf(__ldcg(plr + sp), f, Ls);
    }
    Ls = warp_sum(Ls);
    if (lane == 0) {
      s_M[g] = M;
      s_L[g] = Ls;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D, c = idx % D;
    const size_t row = static_cast<size_t>(b) * Hq + h * G + g;
    const float* A = a.pacc + row * kMaxSplits * D + c;
    float o0 = 0.f, o1 = 0.f;
    int sp = 0;
    for (; sp + 1 < n_split; sp += 2) {
      o0 = fmaf(__ldcg(A + sp * D), s_w[g * kMaxSplits + sp], o0);
      o1 = fmaf(__ldcg(A + (sp + 1) * D), s_w[g * kMaxSplits + sp + 1], o1);
    }
    if (sp < n_split) o0 = fmaf(__ldcg(A + sp * D), s_w[g * kMaxSplits + sp], o0);
    const float Ls = s_L[g];
    a.out[row * D + c] = Ls > 0.f ? (o0 + o1) / Ls : 0.f;
    if (c == 0 && a.lse) a.lse[row] = Ls > 0.f ? (s_M[g] + log2f(Ls)) * kLn2 : -INFINITY;
  }
  if (threadIdx.x == 0) a.counters[unit] = 0;  // ready for the next call
}

template <typename T, typename TQ, int D, int G>
cudaError_t attn_typed(const spg_params& p, const AttnArgs& a0, int pages_upper, float* out,
                       float* lse, cudaStream_t st) {
  constexpr int threads = (kConsumerWarps + 1) * 32;
  constexpr bool MMA = !is_i8<T>() || (D == 128 && std::is_same<TQ, __half>::value);
  AttnArgs a = a0;
  const int S = p.page_size;
  const int units = p.batch * p.num_kv_heads;
  // a page's K tile must start 1024-byte aligned for the swizzled TMA tiles
  const uint32_t pb = MMA ? (kv_stage_bytes<T, D>(S) + 1023u) & ~1023u : kv_stage_bytes<T, D>(S);
  int pps = 1;
  while (pps * 2 <= kMaxPagesPerStage && (pps * 2) * pb <= static_cast<uint32_t>(kStageBytesTarget))
    pps *= 2;
  const uint32_t sb = pps * pb;
  // a multiple of the consumer warps: each ring slot has one owner
  int stages = max(2, min(kMaxStages, static_cast<int>(kRingBytesTarget / sb)));
  stages = (stages + kConsumerWarps - 1) / kConsumerWarps * kConsumerWarps;
  if (stages > kMaxStages) return cudaErrorNotSupported;
  a.stages = stages;
  a.pages_per_stage = pps;
  a.stage_bytes = sb;
  a.page_bytes = pb;
  if constexpr (MMA) {
    const long long rows = static_cast<long long>(p.num_phys_pages) * p.num_kv_heads * S;
    bool wk = false, wv = false;
    if (!make_kv_tmap(&a.tmk, a.k_pool, p.kv_dtype, rows, D, S, &wk) ||
        !make_kv_tmap(&a.tmv, a.v_pool, p.kv_dtype, rows, D, S, &wv) || wk != wv)
      return cudaErrorNotSupported;
    a.whole_page = wk ? 1 : 0;
  }
  auto kern = k_attn<T, TQ, D, G>;
  const size_t ring = static_cast<size_t>(stages) * sb;
  const size_t bars = sizeof(uint64_t) * 2 * kMaxStages +
                      sizeof(int) * (kMaxStages + kMaxStages * kMaxPagesPerStage);
  const size_t merge = sizeof(float) * kConsumerWarps * G * (D + 2);
  const size_t comb = sizeof(float) * (G * kMaxSplits + 2 * G);
  const size_t smem = 1024 + max(ring + bars, max(merge, comb));  // + alignment slack
  if (smem > 227u * 1024u) return cudaErrorNotSupported;
  cudaError_t e = ensure_smem(kern, smem);
  if (e != cudaSuccess) return e;
  // one wave: as many CTAs as fit on the GPU at once, spread over the units
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int slots = device_sm_count() * per_sm;
  a.out = out;
  a.lse = lse;
  a.units = units;
  if (!a.sel) {
    // dense: the length plan over one wave (at least two CTAs per unit, so
    // that N >= units); the sum of the parts is at most N + units CTAs
    const int n_cta = max(slots, 2 * units);
    a.planned = 1;
    a.plan_n = n_cta - units;
    a.pages_per_split = 0;
    return launch_pdl(kern, dim3(n_cta, 1), dim3(threads), smem, st, a);
  }
  int n_split = max(1, slots / units);
  n_split = min(n_split, min(kMaxSplits, max(pages_upper, 1)));
  const int pps_split = (max(pages_upper, 1) + n_split - 1) / n_split;
  n_split = max(1, (max(pages_upper, 1) + pps_split - 1) / pps_split);
  a.pages_per_split = pps_split;
  a.planned = 0;
  return launch_pdl(kern, dim3(n_split, units), dim3(threads), smem, st, a);
}

template <typename T, typename TQ>
cudaError_t attn_dispatch_dg(const spg_params& p, const AttnArgs& a, int pages_upper, float* out,
                             float* lse, cudaStream_t st) {
  const int G = p.num_q_heads / p.num_kv_heads;
#define SPG_AT(D_, G_) \
  if (p.head_dim == D_ && G == G_) return attn_typed<T, TQ, D_, G_>(p, a, pages_upper, out, lse, st);
  SPG_AT(128, 1) SPG_AT(128, 2) SPG_AT(128, 4) SPG_AT(128, 8)
  SPG_AT(64, 1) SPG_AT(64, 2) SPG_AT(64, 4) SPG_AT(64, 8)
#undef SPG_AT
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attention(const spg_params& p, const void* q, const void* k_pool,
                             const void* v_pool, const void* k_scale, const void* v_scale,
                             const int32_t* page_table, const int32_t* seq_lens,
                             const int32_t* sel, const int32_t* sel_cnt, float* out, float* lse,
                             const Workspace& ws, cudaStream_t stream) {
  AttnArgs a{};
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.k_scale = static_cast<const __half*>(k_scale);
  a.v_scale = static_cast<const __half*>(v_scale);
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.sel = sel;
  a.sel_cnt = sel_cnt;
  a.pm = ws.pm;
  a.pl = ws.pl;
  a.pacc = ws.pacc;
  a.counters = ws.counters;
  a.hook = ws.hook;
  a.err = ws.err;
  a.Hkv = p.num_kv_heads;
  a.S = p.page_size;
  a.MP = p.max_pages_per_seq;
  a.n_phys = p.num_phys_pages;
  a.n_sel = sel ? n_sel_pages(p) : 0;
  const float scale = p.softmax_scale > 0.f ? p.softmax_scale
                                            : 1.0f / sqrtf(static_cast<float>(p.head_dim));
  a.scale_log2 = scale * kLog2e;
  const int pages_upper = sel ? n_sel_pages(p) : p.max_pages_per_seq;
  switch (p.kv_dtype) {
    case SPG_F16:
      return attn_dispatch_dg<__half, __half>(p, a, pages_upper, out, lse, stream);
    case SPG_BF16:
      return attn_dispatch_dg<__nv_bfloat16, __nv_bfloat16>(p, a, pages_upper, out, lse, stream);
    default:
      if (p.q_dtype == SPG_F16)
        return attn_dispatch_dg<int8_t, __half>(p, a, pages_upper, out, lse, stream);
      return attn_dispatch_dg<int8_t, __nv_bfloat16>(p, a, pages_upper, out, lse, stream);
  }
}

}  // namespace spg
