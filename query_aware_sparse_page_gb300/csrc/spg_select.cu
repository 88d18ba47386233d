// Page scoring and exact top-k page selection.
//
// Scoring streams one metadata row per candidate page:
//  * Quest (Quest 完全拆解, 核心机制): score = max over the kv-head group's
//    query heads of sum_i max(q_i m_i, q_i M_i).  Since M_i >= m_i the max is
//    q_i * (q_i >= 0 ? M_i : m_i); the fp16/bf16 product is exact in fp32,
//    only the channel sum rounds.  A half-warp covers one 2*d*2-byte row
//    with 16-byte loads; a CTA handles 64 pages of one (batch, kv-head).
//  * Sketch (SALS长序列推理优化, QSI steps 1-3): the group-mean query is
//    projected through P and quantised to int8 (same fp32 rule as the keys),
//    the int4 key codes are unpacked to int8 lanes and dotted with dp4a
//    (exact int32), dequantised by sq * sk_block / sqrt(d), and reduced to a
//    block log-sum-exp with warp shuffles.
//
// Top-k (SALS QSI Top-k: exact, stable; Day 10·2: lower index wins ties):
// one CTA per (batch, kv-head) holds the candidates' order-preserving uint32
// keys in shared memory, finds the k-th largest key with a 4 x 8-bit radix
// select, then compacts keys above it plus the lowest-index keys equal to it
// in index order (two block scans), which yields ascending page ids without
// a sort.  Only int32 page ids reach global memory.
#include <float.h>

#include "spg_common.cuh"
#include "spg_internal.h"

namespace spg {
namespace {

constexpr int kScorePagesPerCta = 64;

template <typename T>
__device__ __forceinline__ void unpack2(uint32_t w, float& a, float& b);
template <>
__device__ __forceinline__ void unpack2<__half>(uint32_t w, float& a, float& b) {
  float2 f = __half22float2(*reinterpret_cast<__half2*>(&w));
  a = f.x;
  b = f.y;
}
template <>
__device__ __forceinline__ void unpack2<__nv_bfloat16>(uint32_t w, float& a, float& b) {
  a = __uint_as_float(w << 16);
  b = __uint_as_float(w & 0xffff0000u);
}

template <typename T, int CPL>
__device__ __forceinline__ void load_row_chunk(const T* p, uint32_t (&w)[CPL / 2]) {
  if constexpr (CPL == 8) {
    uint4 r = __ldg(reinterpret_cast<const uint4*>(p));
    w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
  } else {
    uint2 r = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = r.x; w[1] = r.y;
  }
}

// Quest scores: grid (ceil(MP/64), B*Hkv), 256 threads (8 warps x 2 pages x 4).
template <typename T, int D, int G>
__global__ void __launch_bounds__(256) k_quest_score(
    const T* __restrict__ q, const int32_t* __restrict__ page_table,
    const int32_t* __restrict__ seq_lens, const T* __restrict__ minmax, float* __restrict__ scores,
    int Hkv, int S, int MP, int n_phys, int n_sink, int n_recent, int32_t* __restrict__ err) {
  constexpr int CPL = D / 16;  // channels per lane; 16 lanes cover one row
  constexpr int ITER = kScorePagesPerCta / 16;  // page pairs per warp
  __shared__ int s_phys[kScorePagesPerCta];

  const int unit = blockIdx.y;
  const int b = unit / Hkv, h = unit % Hkv;
  const int p0 = blockIdx.x * kScorePagesPerCta;
  int L = seq_lens[b];
  if (L < 0 || L > MP * S) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(err, SPG_DEVERR_SEQ_LEN);
    L = 0;
  }
  const int P = (L + S - 1) / S;
  const int lo = min(n_sink, P), hi = max(P - n_recent, lo);

  for (int i = threadIdx.x; i < kScorePagesPerCta; i += blockDim.x) {
    const int p = p0 + i;
    int ph = -1;
    if (p >= lo && p < hi) {
      ph = page_table[(size_t)b * MP + p];
      if (ph < 0 || ph >= n_phys) {
        record_error(err, SPG_DEVERR_PAGE_ID);
        ph = -1;
      }
    }
    s_phys[i] = ph;
  }

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane >> 4, hl = lane & 15;
  float qf[G][CPL];
  const T* qb = q + ((size_t)b * Hkv * G + (size_t)h * G) * D + hl * CPL;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    uint32_t w[CPL / 2];
    load_row_chunk<T, CPL>(qb + (size_t)g * D, w);
#pragma unroll
    for (int c = 0; c < CPL / 2; ++c) unpack2<T>(w[c], qf[g][2 * c], qf[g][2 * c + 1]);
  }
  __syncthreads();

  uint32_t wm[ITER][CPL / 2], wM[ITER][CPL / 2];
  int phs[ITER];
#pragma unroll
  for (int it = 0; it < ITER; ++it) {
    const int slot = warp * (2 * ITER) + it * 2 + half;
    phs[it] = s_phys[slot];
    if (phs[it] >= 0) {
      const T* row = minmax + ((size_t)phs[it] * Hkv + h) * 2 * D + hl * CPL;
      load_row_chunk<T, CPL>(row, wm[it]);
      load_row_chunk<T, CPL>(row + D, wM[it]);
    } else {
#pragma unroll
      for (int c = 0; c < CPL / 2; ++c) wm[it][c] = wM[it][c] = 0u;
    }
  }
#pragma unroll
  for (int it = 0; it < ITER; ++it) {
    float mf[CPL], Mf[CPL];
#pragma unroll
    for (int c = 0; c < CPL / 2; ++c) {
      unpack2<T>(wm[it][c], mf[2 * c], mf[2 * c + 1]);
      unpack2<T>(wM[it][c], Mf[2 * c], Mf[2 * c + 1]);
    }
    float best = -FLT_MAX;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc = fmaf(qf[g][c], qf[g][c] >= 0.f ? Mf[c] : mf[c], acc);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      best = fmaxf(best, acc);
    }
    const int slot = warp * (2 * ITER) + it * 2 + half;
    const int p = p0 + slot;
    if (hl == 0 && p < MP) scores[(size_t)unit * MP + p] = phs[it] >= 0 ? best : -INFINITY;
  }
}

// int4 nibbles of one 32-bit word -> two words of 4 signed int8 lanes
// (even-index codes, odd-index codes)
__device__ __forceinline__ void unpack_int4x8(uint32_t w, int& even, int& odd) {
  const uint32_t lo = (w & 0x0f0f0f0fu) ^ 0x08080808u;
  const uint32_t hi = ((w >> 4) & 0x0f0f0f0fu) ^ 0x08080808u;
  even = static_cast<int>(__vsub4(lo, 0x08080808u));
  odd = static_cast<int>(__vsub4(hi, 0x08080808u));
}

__device__ __forceinline__ int pack_i8x4(int a, int b, int c, int d) {
  return (a & 0xff) | ((b & 0xff) << 8) | ((c & 0xff) << 16) | ((d & 0xff) << 24);
}

// Sketch scores: grid (ceil(MP/8), B*Hkv), 256 threads, one warp per block.
// ds = 16 (8 bytes of codes per token).
template <typename TQ>
__global__ void __launch_bounds__(256) k_sketch_score(
    const TQ* __restrict__ q, const int32_t* __restrict__ page_table,
    const int32_t* __restrict__ seq_lens, const uint8_t* __restrict__ sketch,
    const float* __restrict__ sketch_scale, const float* __restrict__ proj,
    float* __restrict__ scores, int Hkv, int G, int S, int d, int MP, int n_phys, int n_sink,
    int n_recent, float inv_sqrt_d, int32_t* __restrict__ err) {
  constexpr int DS = 16;
  __shared__ float s_qbar[256];
  __shared__ float s_P[256 * DS];
  __shared__ int s_qc[4];  // packed int8 codes: even 0-6, odd 1-7, even 8-14, odd 9-15
  __shared__ float s_sq;

  const int unit = blockIdx.y;
  const int b = unit / Hkv, h = unit % Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int blk = blockIdx.x * nw + warp;
  int L = seq_lens[b];
  if (L < 0 || L > MP * S) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(err, SPG_DEVERR_SEQ_LEN);
    L = 0;
  }
  const int P = (L + S - 1) / S;
  const int lo = min(n_sink, P), hi = max(P - n_recent, lo);
  int ph = -1;
  if (blk >= lo && blk < hi) {
    ph = page_table[(size_t)b * MP + blk];
    if (ph < 0 || ph >= n_phys) {
      if (lane == 0) record_error(err, SPG_DEVERR_PAGE_ID);
      ph = -1;
    }
  }

  // index query (group mean -> projection -> int8), fp32, fixed order, unfused
  const TQ* qb = q + ((size_t)b * Hkv * G + (size_t)h * G) * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float s = to_f32(qb[i]);
    for (int g = 1; g < G; ++g) s = __fadd_rn(s, to_f32(qb[(size_t)g * d + i]));
    s_qbar[i] = __fdiv_rn(s, static_cast<float>(G));
  }
  for (int i = threadIdx.x; i < d * DS; i += blockDim.x) s_P[i] = proj[i];
  __syncthreads();
  if (warp == 0) {
    float qt = 0.f;
    if (lane < DS)
      for (int i = 0; i < d; ++i) qt = __fadd_rn(qt, __fmul_rn(s_qbar[i], s_P[i * DS + lane]));
    float a = fabsf(qt);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float sq = a > 0.f ? __fdiv_rn(a, 127.0f) : 1.0f;
    int qc = max(-127, min(127, static_cast<int>(rintf(__fdiv_rn(qt, sq)))));
    // gather codes into packed words
    int c[DS];
#pragma unroll
    for (int j = 0; j < DS; ++j) c[j] = __shfl_sync(0xffffffffu, qc, j);
    if (lane == 0) {
      s_qc[0] = pack_i8x4(c[0], c[2], c[4], c[6]);
      s_qc[1] = pack_i8x4(c[1], c[3], c[5], c[7]);
      s_qc[2] = pack_i8x4(c[8], c[10], c[12], c[14]);
      s_qc[3] = pack_i8x4(c[9], c[11], c[13], c[15]);
      s_sq = sq;
    }
  }
  __syncthreads();
  if (blk >= MP) return;
  float* out = scores + (size_t)unit * MP + blk;
  if (ph < 0) {
    if (lane == 0) *out = -INFINITY;
    return;
  }
  const size_t row0 = ((size_t)ph * Hkv + h) * S;
  const float c = __fmul_rn(__fmul_rn(s_sq, sketch_scale[(size_t)ph * Hkv + h]), inv_sqrt_d);
  const int qe0 = s_qc[0], qo0 = s_qc[1], qe1 = s_qc[2], qo1 = s_qc[3];
  float zmax = -INFINITY;
  float z[4];  // up to 128 tokens per block
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int t = lane + 32 * k;
    z[k] = -INFINITY;
    if (t < S) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(sketch + (row0 + t) * (DS / 2)));
      int e0, o0, e1, o1;
      unpack_int4x8(w.x, e0, o0);
      unpack_int4x8(w.y, e1, o1);
      int dot = __dp4a(e0, qe0, 0);
      dot = __dp4a(o0, qo0, dot);
      dot = __dp4a(e1, qe1, dot);
      dot = __dp4a(o1, qo1, dot);
      z[k] = static_cast<float>(dot) * c;
      zmax = fmaxf(zmax, z[k]);
    }
  }
  zmax = warp_max(zmax);
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (lane + 32 * k < S) sum += expf(z[k] - zmax);
  sum = warp_sum(sum);
  if (lane == 0) *out = zmax + logf(sum);
}

// ---- block-wide exclusive scan of one int per thread -----------------------
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* s_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < nw) s_warp[lane] = wi - w;
    if (lane == 31) *s_total = wi;
  }
  __syncthreads();
  const int r = s_warp[warp] + incl - v;
  __syncthreads();
  return r;
}

// Top-k: one CTA (1024 threads) per (batch, kv-head).
__global__ void __launch_bounds__(1024) k_topk(const float* __restrict__ scores,
                                               const int32_t* __restrict__ seq_lens,
                                               int32_t* __restrict__ sel,
                                               int32_t* __restrict__ sel_cnt, int Hkv, int S,
                                               int MP, int n_sel, int n_sink, int n_recent) {
  extern __shared__ uint32_t s_key[];
  __shared__ int s_hist[256];
  __shared__ int s_warp[32];
  __shared__ int s_total;
  __shared__ int s_digit, s_need, s_count;

  const int unit = blockIdx.x;
  const int b = unit / Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int L = seq_lens[b];
  if (L < 0 || L > MP * S) L = 0;  // recorded by the scoring kernel
  const int P = (L + S - 1) / S;
  const int lo = min(n_sink, P), hi = max(P - n_recent, lo);
  const int nc = hi - lo, nf = P - nc;
  const int k_top = min(max(n_sel - nf, 0), nc);
  int32_t* out = sel + (size_t)unit * n_sel;
  const float* srow = scores + (size_t)unit * MP + lo;

  // sinks, then (after the candidates) the recent pages, then -1 padding
  for (int i = tid; i < lo; i += blockDim.x) out[i] = i;
  for (int j = tid; j < P - hi; j += blockDim.x) out[lo + k_top + j] = hi + j;
  const int count = lo + k_top + (P - hi);
  for (int i = count + tid; i < n_sel; i += blockDim.x) out[i] = -1;
  if (tid == 0) sel_cnt[unit] = count;
  if (k_top == 0) return;
  if (k_top == nc) {
    for (int i = tid; i < nc; i += blockDim.x) out[lo + i] = lo + i;
    return;
  }

  for (int i = tid; i < nc; i += blockDim.x) s_key[i] = score_key(srow[i]);
  __syncthreads();

  // radix select of the k_top-th largest key
  uint32_t prefix = 0u, mask = 0u;
  int need = k_top;
  const int n_round = (nc + 31) & ~31;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) s_hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n_round; i += blockDim.x) {
      const uint32_t key = i < nc ? s_key[i] : 0u;
      const bool match = i < nc && (key & mask) == prefix;
      const unsigned act = __ballot_sync(0xffffffffu, match);
      if (match) {
        const int digit = (key >> shift) & 0xff;
        const unsigned peers = __match_any_sync(act, digit);
        if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[digit], __popc(peers));
      }
    }
    __syncthreads();
    if (warp == 0) {
      int c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = s_hist[255 - 8 * lane - j];
        sum += c[j];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      const int excl = incl - sum;
      if (excl < need && incl >= need) {
        int acc = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc + c[j] >= need) {
            s_digit = 255 - 8 * lane - j;
            s_need = need - acc;
            s_count = c[j];
            break;
          }
          acc += c[j];
        }
      }
    }
    __syncthreads();
    const int digit = s_digit;
    need = s_need;
    const int cnt = s_count;
    prefix |= static_cast<uint32_t>(digit) << shift;
    mask |= 0xffu << shift;
    __syncthreads();
    if (cnt == need) break;  // every key of this bucket is taken
  }

  // compaction in index order: keys above the threshold bucket, plus the
  // first `need` keys inside it (lower page index wins ties)
  const int seg = (nc + blockDim.x - 1) / blockDim.x;
  const int i0 = min(tid * seg, nc), i1 = min(i0 + seg, nc);
  int n_eq = 0, n_gt = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t k = s_key[i] & mask;
    n_eq += (k == prefix);
    n_gt += (k > prefix);
  }
  const int eq_base = block_exclusive_scan(n_eq, s_warp, &s_total);
  const int eq_take = min(max(need - eq_base, 0), n_eq);
  const int pos0 = block_exclusive_scan(n_gt + eq_take, s_warp, &s_total);
  int r = eq_base, pos = pos0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t k = s_key[i] & mask;
    bool take = k > prefix;
    if (k == prefix) {
      take = r < need;
      ++r;
    }
    if (take) out[lo + pos++] = lo + i;
  }
}

template <typename T>
cudaError_t quest_score_typed(const spg_params& p, const void* q, const int32_t* pt,
                              const int32_t* lens, const void* minmax, float* scores,
                              int32_t* err, cudaStream_t st) {
  const int G = p.num_q_heads / p.num_kv_heads;
  dim3 grid((p.max_pages_per_seq + kScorePagesPerCta - 1) / kScorePagesPerCta,
            p.batch * p.num_kv_heads);
  const T* qq = static_cast<const T*>(q);
  const T* mm = static_cast<const T*>(minmax);
#define SPG_QS(D_, G_)                                                                          \
  if (p.head_dim == D_ && G == G_) {                                                             \
    k_quest_score<T, D_, G_><<<grid, 256, 0, st>>>(qq, pt, lens, mm, scores, p.num_kv_heads,     \
                                                   p.page_size, p.max_pages_per_seq,            \
                                                   p.num_phys_pages, p.n_sink_pages,            \
                                                   p.n_recent_pages, err);                      \
    return cudaGetLastError();                                                                   \
  }
  SPG_QS(128, 1) SPG_QS(128, 2) SPG_QS(128, 4) SPG_QS(128, 8)
  SPG_QS(64, 1) SPG_QS(64, 2) SPG_QS(64, 4) SPG_QS(64, 8)
#undef SPG_QS
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_score(const spg_params& p, const void* q, const int32_t* page_table,
                         const int32_t* seq_lens, const void* minmax, const uint8_t* sketch,
                         const float* sketch_scale, const float* proj, float* scores,
                         int32_t* err, cudaStream_t stream) {
  if (p.selector == SPG_SEL_QUEST) {
    if (p.kv_dtype == SPG_F16)
      return quest_score_typed<__half>(p, q, page_table, seq_lens, minmax, scores, err, stream);
    return quest_score_typed<__nv_bfloat16>(p, q, page_table, seq_lens, minmax, scores, err,
                                            stream);
  }
  const int G = p.num_q_heads / p.num_kv_heads;
  const int wpb = 8;
  dim3 grid((p.max_pages_per_seq + wpb - 1) / wpb, p.batch * p.num_kv_heads);
  const float inv = 1.0f / sqrtf(static_cast<float>(p.head_dim));
  if (p.q_dtype == SPG_F16)
    k_sketch_score<__half><<<grid, wpb * 32, 0, stream>>>(
        static_cast<const __half*>(q), page_table, seq_lens, sketch, sketch_scale, proj, scores,
        p.num_kv_heads, G, p.page_size, p.head_dim, p.max_pages_per_seq, p.num_phys_pages,
        p.n_sink_pages, p.n_recent_pages, inv, err);
  else
    k_sketch_score<__nv_bfloat16><<<grid, wpb * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(q), page_table, seq_lens, sketch, sketch_scale, proj,
        scores, p.num_kv_heads, G, p.page_size, p.head_dim, p.max_pages_per_seq,
        p.num_phys_pages, p.n_sink_pages, p.n_recent_pages, inv, err);
  return cudaGetLastError();
}

cudaError_t launch_topk(const spg_params& p, const float* scores, const int32_t* seq_lens,
                        int32_t* sel, int32_t* sel_cnt, int32_t* err, cudaStream_t stream) {
  (void)err;
  const size_t smem = sizeof(uint32_t) * (size_t)p.max_pages_per_seq;
  static int configured_bytes = 0;
  if (smem > 48 * 1024 && (int)smem > configured_bytes) {
    cudaError_t e = cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(uint32_t) * kMaxTopkPages));
    if (e != cudaSuccess) return e;
    configured_bytes = (int)(sizeof(uint32_t) * kMaxTopkPages);
  }
  k_topk<<<p.batch * p.num_kv_heads, 1024, smem, stream>>>(
      scores, seq_lens, sel, sel_cnt, p.num_kv_heads, p.page_size, p.max_pages_per_seq,
      n_sel_pages(p), p.n_sink_pages, p.n_recent_pages);
  return cudaGetLastError();
}

}  // namespace spg
