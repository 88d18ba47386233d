// Pieces of page scoring and exact top-k shared by the scoring kernels and
// the fused single-launch decode step.
//
// Quest bound (Quest 完全拆解, 核心机制): sum_i max(q_i m_i, q_i M_i), the max
// over the kv-head group's query heads; since M_i >= m_i the max is
// q_i * (q_i >= 0 ? M_i : m_i), exact in fp32 for fp16/bf16 inputs, so only
// the channel sum rounds.  Sketch scores (SALS长序列推理优化, QSI steps 1-3).
// Exact top-k with lower index winning ties (SALS QSI Top-k; Day 10·2
// 确定性红线): see block_topk.
#pragma once

#include <float.h>

#include "spg_common.cuh"

namespace spg {

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

struct TopkShared {
  int hist[2048];
  int warp_tot[32];
  int total;
  int digit, need, cnt;
  uint32_t kmin, kmax;
};

// Exact top-k of keys[0, n) (shared memory), larger key first, lower index
// first among equal keys; writes the chosen indices + base, ascending, to
// dst[0, k).  0 < k < n.  Every thread of the block calls it.
inline __device__ void block_topk(const uint32_t* keys, int n, int k, int base, int32_t* dst,
                           TopkShared& t) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int nw = nt >> 5;
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int i = tid; i < n; i += nt) {
    const uint32_t x = keys[i];
    mn = min(mn, x);
    mx = max(mx, x);
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    t.hist[warp] = static_cast<int>(mn);
    t.hist[32 + warp] = static_cast<int>(mx);
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t a = lane < nw ? static_cast<uint32_t>(t.hist[lane]) : 0xffffffffu;
    uint32_t c = lane < nw ? static_cast<uint32_t>(t.hist[32 + lane]) : 0u;
    a = __reduce_min_sync(0xffffffffu, a);
    c = __reduce_max_sync(0xffffffffu, c);
    if (lane == 0) {
      t.kmin = a;
      t.kmax = c;
    }
  }
  __syncthreads();
  mn = t.kmin;
  mx = t.kmax;
  uint32_t prefix, mask;
  int need = k;
  if (mn == mx) {  // every key equal: the lowest indices win
    prefix = mx;
    mask = 0xffffffffu;
  } else {
    int hb = 31 - __clz(static_cast<int>(mn ^ mx));  // highest bit where keys differ
    mask = ~((2u << hb) - 1u);                         // the bits every key shares
    prefix = mx & mask;
    while (true) {
      const int shift = max(hb - 10, 0);
      const int bins = 1 << (hb - shift + 1);
      for (int i = tid; i < bins; i += nt) t.hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < n; i += nt) {
        const uint32_t x = keys[i];
        if ((x & mask) == prefix) atomicAdd(&t.hist[(x >> shift) & (bins - 1)], 1);
      }
      __syncthreads();
      // bins in descending order, a contiguous run per thread
      const int bpt = (bins + nt - 1) / nt;
      const int top = bins - 1 - tid * bpt;
      int local = 0;
      for (int j = 0; j < bpt; ++j)
        if (top - j >= 0) local += t.hist[top - j];
      const int excl = block_exclusive_scan(local, t.warp_tot, &t.total);
      if (excl < need && excl + local >= need) {
        int acc = excl;
        for (int j = 0; j < bpt; ++j) {
          const int c = t.hist[top - j];
          if (acc + c >= need) {
            t.digit = top - j;
            t.need = need - acc;
            t.cnt = c;
            break;
          }
          acc += c;
        }
      }
      __syncthreads();
      const int digit = t.digit, cnt = t.cnt;
      need = t.need;
      prefix |= static_cast<uint32_t>(digit) << shift;
      mask |= static_cast<uint32_t>(bins - 1) << shift;
      __syncthreads();
      if (cnt == need || shift == 0) break;  // the whole bucket is taken, or keys are exact
      hb = shift - 1;
    }
  }
  // compaction in index order: keys above the threshold bucket, plus the
  // first `need` keys inside it
  const int seg = (n + nt - 1) / nt;
  const int i0 = min(tid * seg, n), i1 = min(i0 + seg, n);
  int n_eq = 0, n_gt = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t x = keys[i] & mask;
    n_eq += (x == prefix);
    n_gt += (x > prefix);
  }
  const int eq_base = block_exclusive_scan(n_eq, t.warp_tot, &t.total);
  const int eq_take = min(max(need - eq_base, 0), n_eq);
  int pos = block_exclusive_scan(n_gt + eq_take, t.warp_tot, &t.total);
  int r = eq_base;
  for (int i = i0; i < i1; ++i) {
    const uint32_t x = keys[i] & mask;
    bool take = x > prefix;
    if (x == prefix) {
      take = r < need;
      ++r;
    }
    if (take) dst[pos++] = base + i;
  }
}


// Quest bound of one page for the group's G query rows: a half-warp holds
// CPL = D/16 channels of the row per lane (wm / wM: m and M as packed
// 16-bit pairs); every lane of the half-warp returns the group's score.
template <typename T, int D, int G>
__device__ __forceinline__ float quest_bound(const float (&qf)[G][D / 16], const uint32_t* wm,
                                             const uint32_t* wM) {
  constexpr int CPL = D / 16;
  float mf[CPL], Mf[CPL];
#pragma unroll
  for (int c = 0; c < CPL / 2; ++c) {
    unpack2<T>(wm[c], mf[2 * c], mf[2 * c + 1]);
    unpack2<T>(wM[c], Mf[2 * c], Mf[2 * c + 1]);
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
  return best;
}

// ---- Quest bound on tensor cores -------------------------------------------
// With q- = min(q, 0) and q+ = max(q, 0), max(q m, q M) = q- m + q+ M exactly
// (M >= m), so the bounds of a tile of 16 pages for the G query rows of a
// group are one [16 x 2d] x [2d x G] product: A = the tile's metadata rows
// (m then M, staged in shared memory), B = [q-; q+] (G columns, zero-padded
// to 8).  mma.sync m16n8k16 with fp16/bf16 operands (q-/q+ are q or 0, so
// exact) and fp32 accumulation; ldmatrix reads the chunk-swizzled rows
// without bank conflicts.  The group score of a page is the max over its G
// columns.  (ldmatrix_x4 / mma_16816: spg_common.cuh)
template <typename T, int D, int G>
struct QuestMma {
  static constexpr int KS = 2 * D / 16;  // k-steps over m then M
  uint32_t bf[KS][2];                    // B fragments (q-; q+), one column per query row

  // qrows: the group's G query rows (global); lane layout of the B fragment:
  // column n = lane / 4, k pairs (2t, 2t+1) and (2t+8, 2t+9), t = lane % 4
  __device__ void init(const T* qrows, int lane) {
    const int n = lane >> 2, t = lane & 3;
    const T zero = static_cast<T>(0.f);
#pragma unroll
    for (int j = 0; j < KS; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        T v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int k = 16 * j + 2 * t + 8 * hf + e;
          v[e] = zero;
          if (n < G) {
            const T qv = qrows[n * D + (k < D ? k : k - D)];
            const float f = to_f32(qv);
            v[e] = (k < D) ? (f < 0.f ? qv : zero) : (f > 0.f ? qv : zero);
          }
        }
        bf[j][hf] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&v[0])) |
                    (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&v[1])) << 16);
      }
  }

  // 16 pages whose rows start at `rows` (shared memory, row stride 2d), the
  // first being logical page p0.  Lanes with lane % 4 == 0 return the group
  // score of tile row lane/4 in s0 and of row lane/4 + 8 in s1.
  __device__ void tile(const T* rows, int p0, int lane, float& s0, float& s1) const {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    const int mi = lane >> 3, r = (mi & 1) * 8 + (lane & 7);
    const int key = (p0 + r) & 7;
    const uint32_t base = smem_u32(rows + r * 2 * D);
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      uint32_t a[4];
      ldmatrix_x4(a, base + ((((2 * j) + (mi >> 1)) ^ key) << 4));
      mma_16816<T>(c, a, bf[j][0], bf[j][1]);
    }
    const int t = lane & 3;
    float m0 = -FLT_MAX, m1 = -FLT_MAX;
    if (2 * t < G) {
      m0 = c[0];
      m1 = c[2];
    }
    if (2 * t + 1 < G) {
      m0 = fmaxf(m0, c[1]);
      m1 = fmaxf(m1, c[3]);
    }
    if constexpr (G > 2) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
    }
    if constexpr (G > 4) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
    }
    s0 = m0;
    s1 = m1;
  }
};

// the group's query rows for the lane's CPL channels (half-warp layout)
template <typename T, int D, int G>
__device__ __forceinline__ void quest_query(const T* qrows, int hl, float (&qf)[G][D / 16]) {
  constexpr int CPL = D / 16;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    uint32_t w[CPL / 2];
    load_row_chunk<T, CPL>(qrows + g * D + hl * CPL, w);
#pragma unroll
    for (int c = 0; c < CPL / 2; ++c) unpack2<T>(w[c], qf[g][2 * c], qf[g][2 * c + 1]);
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


// Index query of the sketch selector for one kv-head group: the group mean
// of the G query rows, projected through P (d x 16) and quantised to int8,
// all in fp32 with one rounded product and one rounded add per step, in
// channel order (the same rule as the key side).  Called by a whole CTA;
// s_qbar holds d floats, s_P d*16 floats.  Leaves the codes packed for dp4a
// in s_qc[4] (even 0-6, odd 1-7, even 8-14, odd 9-15) and the scale in *s_sq.
template <typename TQ>
__device__ void sketch_index_query(const TQ* qb, int G, int d, const float* proj, float* s_qbar,
                                   float* s_P, int* s_qc, float* s_sq) {
  constexpr int DS = 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float s = to_f32(qb[i]);
    for (int g = 1; g < G; ++g) s = __fadd_rn(s, to_f32(qb[static_cast<size_t>(g) * d + i]));
    s_qbar[i] = __fdiv_rn(s, static_cast<float>(G));
  }
  for (int i = threadIdx.x; i < d * DS; i += blockDim.x) s_P[i] = proj[i];
  __syncthreads();
  if (warp == 0) {
    float qt = 0.f;
    if (lane < DS)
      for (int i = 0; i < d; ++i) qt = __fadd_rn(qt, __fmul_rn(s_qbar[i], s_P[i * DS + lane]));
    float am = fabsf(qt);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const float sq = am > 0.f ? __fdiv_rn(am, 127.0f) : 1.0f;
    const int qc = max(-127, min(127, static_cast<int>(rintf(__fdiv_rn(qt, sq)))));
    int c[DS];
#pragma unroll
    for (int j = 0; j < DS; ++j) c[j] = __shfl_sync(0xffffffffu, qc, j);
    if (lane == 0) {
      s_qc[0] = pack_i8x4(c[0], c[2], c[4], c[6]);
      s_qc[1] = pack_i8x4(c[1], c[3], c[5], c[7]);
      s_qc[2] = pack_i8x4(c[8], c[10], c[12], c[14]);
      s_qc[3] = pack_i8x4(c[9], c[11], c[13], c[15]);
      *s_sq = sq;
    }
  }
  __syncthreads();
}

// Block log-sum-exp score of one block of S <= 128 tokens, computed by a
// whole warp; wk[k] holds token lane + 32k's 8 bytes of int4 codes.
__device__ __forceinline__ float sketch_block_score(const uint2 (&wk)[4], int S, const int* qc,
                                                    float cz) {
  const int lane = threadIdx.x & 31;
  float zmax = -INFINITY;
  float z[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    z[k] = -INFINITY;
    if (lane + 32 * k < S) {
      int e0, o0, e1, o1;
      unpack_int4x8(wk[k].x, e0, o0);
      unpack_int4x8(wk[k].y, e1, o1);
      int dot = __dp4a(e0, qc[0], 0);
      dot = __dp4a(o0, qc[1], dot);
      dot = __dp4a(e1, qc[2], dot);
      dot = __dp4a(o1, qc[3], dot);
      z[k] = static_cast<float>(dot) * cz;
      zmax = fmaxf(zmax, z[k]);
    }
  }
  zmax = warp_max(zmax);
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (lane + 32 * k < S) sum += expf(z[k] - zmax);
  sum = warp_sum(sum);
  return zmax + logf(sum);
}

}  // namespace spg
