// Split-K flash-decoding over gathered KV pages, and the log-sum-exp combine.
//
// Sources: SALS长序列推理优化, SFAA (QK^T, online softmax, P@V, rescale over
// the selected K/V; int8 K/V dequantised by their scales) and AICPU Tiling
// challenge 2 (a row split over several cores is merged by a reduction);
// Quest 完全拆解, 三段式 kernel (Approximate attention reads only the top-K
// pages); Day 10·2 (softmax renormalised over the selected blocks only).
//
// Grid = (splits, batch * kv-heads).  A CTA owns a contiguous range of the
// unit's page list (selected ids, or every page for the dense baseline).
// All its threads first resolve the range's logical -> physical page ids
// into shared memory (one round trip for the whole range), then each warp
// runs its own pipeline over every W-th page of the range: lane 0 issues
// cp.async.bulk copies (the TMA bulk engine) of the page's contiguous K and
// V tiles ([S][d] per kv-head in the [P][Hkv][S][d] pool, plus the per-token
// scales for int8) into a STAGES-deep shared-memory ring, completion tracked
// by one mbarrier per stage; the warp computes on CUDA cores with the head
// dimension split across lanes (a K/V row is read once, conflict-free) and
// the G query rows of the kv-head group sharing every tile (GQA).  Every
// barrier wait is bounded; a wait that runs out records SPG_DEVERR_TIMEOUT,
// drains the copies this warp issued (bounded again) and stops.
//
// Partials per (batch, q-head, split): running max m (log2 domain, scale
// folded in), running sum l, unnormalised accumulator acc[d].  The last CTA
// of a unit to arrive (an atomic counter per unit in the workspace, reset by
// that CTA) merges the unit's splits and writes out and lse, so one launch
// does the whole attention.
#include <float.h>

#include "spg_common.cuh"
#include "spg_internal.h"

namespace spg {
namespace {

constexpr int kMaxPagesPerSplit = 1024;

struct AttnArgs {
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
  float* out;
  float* lse;
  int32_t* err;
  int Hkv, S, MP, n_phys, n_sel, pages_per_split;
  float scale_log2;
};

template <typename T>
constexpr bool is_i8() { return sizeof(T) == 1; }

// bytes of one stage: K tile, V tile, and for int8 the two fp16 scale rows
template <typename T, int D>
__host__ __device__ inline uint32_t stage_bytes(int S) {
  const uint32_t tile = static_cast<uint32_t>(S) * D * sizeof(T);
  const uint32_t sc = is_i8<T>() ? static_cast<uint32_t>(S) * 2 : 0u;
  return 2 * tile + 2 * sc;
}

template <typename T, int CPL>
__device__ __forceinline__ void row_f32(const T* p, float* o) {
  if constexpr (CPL == 4) load4_f32<T>(p, o);
  else load2_f32<T>(p, o);
}

template <typename T, typename TQ, int D, int G, int W, int STAGES>
__global__ void __launch_bounds__(W * 32) k_attn(const AttnArgs a) {
  constexpr int CPL = D / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const int S = a.S;
  const uint32_t tile = static_cast<uint32_t>(S) * D * sizeof(T);
  const uint32_t scb = is_i8<T>() ? static_cast<uint32_t>(S) * 2 : 0u;
  const uint32_t sbytes = stage_bytes<T, D>(S);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + static_cast<size_t>(warp) * STAGES * sbytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(W) * STAGES * sbytes) +
                   warp * STAGES;
  int2* s_pg = reinterpret_cast<int2*>(smem + static_cast<size_t>(W) * STAGES * sbytes +
                                       sizeof(uint64_t) * W * STAGES);

  const int unit = blockIdx.y, split = blockIdx.x;
  const int Hkv = a.Hkv;
  const int b = unit / Hkv, h = unit % Hkv;
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
  const int s0 = split * a.pages_per_split;
  const int s1 = min(s0 + a.pages_per_split, count);
  const int n_range = max(s1 - s0, 0);

  // resolve the range's pages: (physical page or -1, valid tokens)
  for (int i = threadIdx.x; i < n_range; i += blockDim.x) {
    const int idx = s0 + i;
    int lp = a.sel ? a.sel[static_cast<size_t>(unit) * a.n_sel + idx] : idx;
    int ph = -1, nv = 0;
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
    s_pg[i] = make_int2(ph, nv);
  }
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  __syncthreads();

  // query rows of the group, pre-scaled into the log2 domain
  const int Hq = Hkv * G;
  const TQ* qb = static_cast<const TQ*>(a.q) + (static_cast<size_t>(b) * Hq + h * G) * D + lane * CPL;
  float qf[G][CPL], acc[G][CPL], m[G], l[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    row_f32<TQ, CPL>(qb + g * D, qf[g]);
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      qf[g][c] *= a.scale_log2;
      acc[g][c] = 0.f;
    }
    m[g] = -INFINITY;
    l[g] = 0.f;
  }

  const T* kpool = static_cast<const T*>(a.k_pool);
  const T* vpool = static_cast<const T*>(a.v_pool);
  const int nw = n_range > warp ? (n_range - warp + W - 1) / W : 0;
  const uint64_t pol = policy_evict_first();

  auto issue = [&](int j) {
    const int stage = j % STAGES;
    const int2 pg = s_pg[warp + W * j];
    uint8_t* dst = ring + static_cast<size_t>(stage) * sbytes;
    if (pg.x < 0) {
      mbar_arrive_expect_tx(&bars[stage], 0);
      return;
    }
    const size_t ph = static_cast<size_t>(pg.x) * Hkv + h;
    mbar_arrive_expect_tx(&bars[stage], sbytes);
    bulk_g2s_hint(dst, kpool + ph * S * D, tile, &bars[stage], pol);
    bulk_g2s_hint(dst + tile, vpool + ph * S * D, tile, &bars[stage], pol);
    if constexpr (is_i8<T>()) {
      // per-token scale rows, S * 2 bytes (a multiple of 16 since S % 8 == 0)
      bulk_g2s(dst + 2 * tile, a.k_scale + ph * S, scb, &bars[stage]);
      bulk_g2s(dst + 2 * tile + scb, a.v_scale + ph * S, scb, &bars[stage]);
    }
  };

  if (lane == 0)
    for (int j = 0; j < min(STAGES, nw); ++j) issue(j);
  __syncwarp();

  bool timed_out = false;
  for (int j = 0; j < nw; ++j) {
    const int stage = j % STAGES;
    const uint32_t parity = (j / STAGES) & 1;
    if (!mbar_wait_bounded(&bars[stage], parity)) {
      if (lane == 0) record_error(a.err, SPG_DEVERR_TIMEOUT);
      // drain what this warp still has in flight, then stop
      for (int jj = j; jj < min(j + STAGES, nw); ++jj)
        mbar_wait_bounded(&bars[jj % STAGES], (jj / STAGES) & 1);
      timed_out = true;
      break;
    }
    const int2 pg = s_pg[warp + W * j];
    if (pg.x >= 0) {
      const uint8_t* st = ring + static_cast<size_t>(stage) * sbytes;
      const T* Ks = reinterpret_cast<const T*>(st);
      const T* Vs = reinterpret_cast<const T*>(st + tile);
      const __half* ksc = reinterpret_cast<const __half*>(st + 2 * tile);
      const __half* vsc = reinterpret_cast<const __half*>(st + 2 * tile + scb);
      const int nv = pg.y;
      for (int t0 = 0; t0 < nv; t0 += 8) {
        float z[8][G];
#pragma unroll
        for (int tt = 0; tt < 8; ++tt) {
          const int t = t0 + tt;
          if (t < nv) {
            float kf[CPL];
            row_f32<T, CPL>(Ks + t * D + lane * CPL, kf);
            float ksv = 1.f;
            if constexpr (is_i8<T>()) ksv = __half2float(ksc[t]);
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float part = 0.f;
#pragma unroll
              for (int c = 0; c < CPL; ++c) part = fmaf(qf[g][c], kf[c], part);
              z[tt][g] = warp_sum(part) * ksv;
            }
          } else {
#pragma unroll
            for (int g = 0; g < G; ++g) z[tt][g] = -INFINITY;
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float cm = z[0][g];
#pragma unroll
          for (int tt = 1; tt < 8; ++tt) cm = fmaxf(cm, z[tt][g]);
          const float mn = fmaxf(m[g], cm);  // finite: token t0 is valid
          const float corr = exp2f(m[g] - mn);
          l[g] *= corr;
#pragma unroll
          for (int c = 0; c < CPL; ++c) acc[g][c] *= corr;
          m[g] = mn;
#pragma unroll
          for (int tt = 0; tt < 8; ++tt) {
            const float pz = exp2f(z[tt][g] - mn);
            l[g] += pz;
            z[tt][g] = pz;  // reuse as the probability
          }
        }
#pragma unroll
        for (int tt = 0; tt < 8; ++tt) {
          const int t = t0 + tt;
          if (t < nv) {
            float vf[CPL];
            row_f32<T, CPL>(Vs + t * D + lane * CPL, vf);
            float vsv = 1.f;
            if constexpr (is_i8<T>()) vsv = __half2float(vsc[t]);
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float pv = z[tt][g] * vsv;
#pragma unroll
              for (int c = 0; c < CPL; ++c) acc[g][c] = fmaf(pv, vf[c], acc[g][c]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && j + STAGES < nw) {
      fence_proxy_async();
      issue(j + STAGES);
    }
    __syncwarp();
  }
  (void)timed_out;

  // merge the W warps of this CTA (reusing the ring), then write the partial
  __syncthreads();
  float* s_m = reinterpret_cast<float*>(smem);          // [W][G]
  float* s_l = s_m + W * G;                              // [W][G]
  float* s_acc = s_l + W * G;                            // [W][G][D]
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      s_m[warp * G + g] = m[g];
      s_l[warp * G + g] = l[g];
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) s_acc[(warp * G + g) * D + lane * CPL + c] = acc[g][c];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D, c = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, s_m[w * G + g]);
    float A = 0.f, Ls = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float f = exp2f(s_m[w * G + g] - M);
        A = fmaf(s_acc[(w * G + g) * D + c], f, A);
        Ls = fmaf(s_l[w * G + g], f, Ls);
      }
    }
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
  __shared__ int s_last;
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(&a.counters[unit], 1);
    s_last = (prev == static_cast<int>(gridDim.x) - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int n_split = gridDim.x;
  for (int g = warp; g < G; g += W) {
    const size_t row = static_cast<size_t>(b) * Hq + h * G + g;
    const float* pmr = a.pm + row * kMaxSplits;
    const float* plr = a.pl + row * kMaxSplits;
    float M = -INFINITY;
    for (int sp = lane; sp < n_split; sp += 32) M = fmaxf(M, __ldcg(pmr + sp));
    M = warp_max(M);
    float o[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) o[c] = 0.f;
    float Ls = 0.f;
    if (M != -INFINITY) {
      for (int sp = 0; sp < n_split; ++sp) {
        const float f = exp2f(__ldcg(pmr + sp) - M);
        Ls = fmaf(__ldcg(plr + sp), f, Ls);
        const float* A = a.pacc + (row * kMaxSplits + sp) * D + lane * CPL;
#pragma unroll
        for (int c = 0; c < CPL; ++c) o[c] = fmaf(__ldcg(A + c), f, o[c]);
      }
    }
    float* orow = a.out + row * D + lane * CPL;
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) orow[c] = o[c] * inv;
    if (a.lse && lane == 0) a.lse[row] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
  }
  if (threadIdx.x == 0) a.counters[unit] = 0;  // ready for the next call
}

template <typename T, typename TQ, int D, int G>
cudaError_t attn_typed(const spg_params& p, const AttnArgs& a0, int pages_upper, float* out,
                       float* lse, cudaStream_t st) {
  constexpr int W = 4;
  constexpr int STAGES = is_i8<T>() ? 2 : 3;
  AttnArgs a = a0;
  const int units = p.batch * p.num_kv_heads;
  const uint32_t sb = stage_bytes<T, D>(p.page_size);
  auto kern = k_attn<T, TQ, D, G, W, STAGES>;
  const size_t ring = static_cast<size_t>(W) * STAGES * sb;
  const size_t merge = sizeof(float) * W * G * (D + 2);
  // split plan: about two CTAs per SM in total, bounded by the workspace
  const int ctas_per_sm = 2;
  const int target = device_sm_count() * ctas_per_sm;
  int n_split = (target + units - 1) / units;
  n_split = max(1, min(n_split, min(kMaxSplits, max(pages_upper, 1))));
  int pps = (max(pages_upper, 1) + n_split - 1) / n_split;
  pps = max(pps, (pages_upper + kMaxSplits - 1) / kMaxSplits);
  if (pps > kMaxPagesPerSplit) return cudaErrorInvalidValue;
  n_split = max(1, (pages_upper + pps - 1) / pps);
  a.pages_per_split = pps;
  const size_t smem = max(ring + sizeof(uint64_t) * W * STAGES + sizeof(int2) * pps, merge);
  static int configured = 0;
  if (smem > 48 * 1024 && static_cast<int>(smem) > configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = static_cast<int>(smem);
  }
  a.out = out;
  a.lse = lse;
  dim3 grid(n_split, units);
  kern<<<grid, W * 32, smem, st>>>(a);
  return cudaGetLastError();
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
