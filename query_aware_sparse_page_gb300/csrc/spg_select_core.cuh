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

#include <climits>
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

// ---- block-wide exclusive scan of one value per thread (int, or uint32
// with wrap-around addition) -----------------------------------------------
template <typename V>
__device__ __forceinline__ V block_exclusive_scan_t(V v, V* s_warp, V* s_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  V incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const V n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    V w = lane < nw ? s_warp[lane] : V(0);
    V wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const V n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < nw) s_warp[lane] = wi - w;
    if (lane == 31) *s_total = wi;
  }
  __syncthreads();
  const V r = s_warp[warp] + incl - v;
  __syncthreads();
  return r;
}

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

// Shared state of the block top-k for up to MAXN keys.
// 16-byte aligned: the histogram is cleared and read with 16-byte accesses
template <int MAXN>
struct alignas(16) TopkSmem {
  static constexpr int kWords = (MAXN + 31) / 32;
  int hist[2048];
  int wa[32], wb[32];
  int total, digit, need, cnt;
  uint32_t kmin, kmax;  // min / max of the keys (set by the caller when it knows them)
  uint32_t thr;         // exact threshold key found among the candidates
  int need_thr;         // keys equal to thr to take, lowest indices first
  int ncand;
  int cand[256];        // indices of the keys in the threshold bucket, when it is small
  uint32_t candk[256];  // and their keys
  uint32_t gtw[kWords];  // bitmap: keys above the threshold
  uint32_t eqw[kWords];  // bitmap: keys in the threshold bucket (or equal to the threshold)
};

// Block-wide search of t.hist[0, 2048) (bins past the pass's bin count are
// zero) for the bin in which the descending cumulative count reaches `need`:
// t.digit, t.need (still needed inside it), t.cnt (its keys).  Thread j < 128
// holds bins [2048 - 16 (j + 1), 2048 - 16 j) in registers (four 16-byte
// loads); one block scan of the per-thread sums finds the thread, which then
// walks its registers.  Every thread calls it.
template <int MAXN>
__device__ __forceinline__ void topk_find_bin(TopkSmem<MAXN>& t, int need) {
  const int tid = threadIdx.x;
  int4 q[4] = {};
  int sum = 0;
  if (tid < 128) {
    const int4* h4 = reinterpret_cast<const int4*>(t.hist);
#pragma unroll
    for (int u = 0; u < 4; ++u) q[u] = h4[511 - 4 * tid - u];
#pragma unroll
    for (int u = 0; u < 4; ++u) sum += q[u].x + q[u].y + q[u].z + q[u].w;
  }
  const int excl = block_exclusive_scan(sum, t.wa, &t.total);
  if (tid < 128 && excl < need && excl + sum >= need) {
    int acc = excl;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v[4] = {q[u].w, q[u].z, q[u].y, q[u].x};  // descending bins
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (acc < need && acc + v[e] >= need) {
          t.digit = 2047 - 16 * tid - 4 * u - e;
          t.need = need - acc;
          t.cnt = v[e];
        }
        acc += v[e];
      }
    }
  }
  __syncthreads();
}

// Chunk u of a run of 16-byte chunks, visited in an order rotated by `rot`:
// threads whose runs start at the same offset modulo 128 bytes but differ in
// `rot` then hit different bank groups on each load.  The caller does not
// depend on the order (or shifts results by the chunk index).
__device__ __forceinline__ uint4 rot_chunk(const uint32_t* p, int u, int rot, int nchunks, int& j) {
  j = (u + rot) & (nchunks - 1);
  return reinterpret_cast<const uint4*>(p)[j];
}

// Exact top-k of keys[0, n) (shared memory, 16-byte aligned, n <= MAXN):
// larger key first, lower index first among equal keys; writes the chosen
// indices + base, ascending, to dst[0, k).  0 < k < n; blockDim.x >= 128.
// Every thread of the block calls it.  minmax_ready: the caller has stored
// the keys' min / max in t.kmin / t.kmax; hist_clear: t.hist is already all
// zeros (both made visible by a barrier).
//
// Radix selection on the order-preserving keys: the bits every key shares
// are skipped and a histogram pass resolves the next 11 bits, as often as it
// takes for the bucket holding the k-th key to be taken whole or to hold at
// most 256 keys.  One pass then records, as bitmaps (a thread per 32 keys),
// the keys above that bucket and the keys in it, gathering the latter when
// there are few; the exact threshold among the gathered keys is found by
// counting, for each, the keys above and equal to it, and the bitmaps are
// corrected.  Warp 0 turns the bitmaps into ascending indices: every key
// above, plus the first `need` keys equal to the threshold.
template <int MAXN>
__device__ __forceinline__ void block_topk(const uint32_t* __restrict__ keys, int n, int k,
                                           int base, int32_t* __restrict__ dst, TopkSmem<MAXN>& t,
                                           bool minmax_ready = false, bool hist_clear = false) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int nw = nt >> 5;
  const int n16 = n & ~15;  // keys in whole 16-key runs; the tail is read one by one
  if (n <= nt) {
    // Few keys: thread i ranks key i by counting the keys that come before it
    // in the total order (key descending, index ascending); the ranks are a
    // permutation of 0 .. n-1 and rank < k is the top-k.  One block scan of
    // the chosen flags gives the ascending positions.
    int r = 0;
    if (tid < n) {
      const uint32_t x = keys[tid];
      const int n4 = n & ~3;
#pragma unroll 4
      for (int j = 0; j < n4; j += 4) {
        const uint4 y = *reinterpret_cast<const uint4*>(keys + j);  // the same 16 bytes for the whole warp
        r += (y.x > x) || (y.x == x && j < tid);
        r += (y.y > x) || (y.y == x && j + 1 < tid);
        r += (y.z > x) || (y.z == x && j + 2 < tid);
        r += (y.w > x) || (y.w == x && j + 3 < tid);
      }
      for (int j = n4; j < n; ++j) {
        const uint32_t y = keys[j];
        r += (y > x) || (y == x && j < tid);
      }
    }
    const bool chosen = tid < n && r < k;
    const int pos = block_exclusive_scan(chosen ? 1 : 0, t.wa, &t.total);
    if (chosen) dst[pos] = base + tid;
    __syncthreads();
    return;
  }
  if (!minmax_ready) {
    uint32_t mn = 0xffffffffu, mx = 0u;
    for (int r = tid; r * 16 < n16; r += nt) {  // runs 64 B apart: rotate by r / 2
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        int j;
        const uint4 v = rot_chunk(keys + r * 16, u, r >> 1, 4, j);
        mn = min(min(mn, min(v.x, v.y)), min(v.z, v.w));
        mx = max(max(mx, max(v.x, v.y)), max(v.z, v.w));
      }
    }
    for (int i = n16 + tid; i < n; i += nt) {
      mn = min(mn, keys[i]);
      mx = max(mx, keys[i]);
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) {
      t.wa[warp] = static_cast<int>(mn);
      t.wb[warp] = static_cast<int>(mx);
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t a = lane < nw ? static_cast<uint32_t>(t.wa[lane]) : 0xffffffffu;
      uint32_t c = lane < nw ? static_cast<uint32_t>(t.wb[lane]) : 0u;
      a = __reduce_min_sync(0xffffffffu, a);
      c = __reduce_max_sync(0xffffffffu, c);
      if (lane == 0) {
        t.kmin = a;
        t.kmax = c;
      }
    }
    __syncthreads();
  }
  const uint32_t mn = t.kmin, mx = t.kmax;
  uint32_t prefix, mask;
  int need = k;
  bool resolve = false;
  if (mn == mx) {  // every key equal: the lowest indices win
    prefix = mx;
    mask = 0xffffffffu;
  } else {
    int hb = 31 - __clz(static_cast<int>(mn ^ mx));  // highest bit where keys differ
    mask = hb == 31 ? 0u : ~((2u << hb) - 1u);         // the bits every key shares
    prefix = mx & mask;
    bool first = true;
    while (true) {
      const int shift = max(hb - 10, 0);
      const int nb = 1 << (hb - shift + 1);
      if (!(first && hist_clear)) {
        for (int i = tid; i < 512; i += nt) reinterpret_cast<int4*>(t.hist)[i] = make_int4(0, 0, 0, 0);
        __syncthreads();
      }
      for (int r = tid; r * 16 < n16; r += nt) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          int j;
          v[u] = rot_chunk(keys + r * 16, u, r >> 1, 4, j);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (first || (x[e] & mask) == prefix) atomicAdd(&t.hist[(x[e] >> shift) & (nb - 1)], 1);
        }
      }
      for (int i = n16 + tid; i < n; i += nt) {
        const uint32_t x = keys[i];
        if (first || (x & mask) == prefix) atomicAdd(&t.hist[(x >> shift) & (nb - 1)], 1);
      }
      __syncthreads();
      topk_find_bin(t, need);
      first = false;
      const int cnt = t.cnt;
      prefix |= static_cast<uint32_t>(t.digit) << shift;
      mask |= static_cast<uint32_t>(nb - 1) << shift;
      need = t.need;
      if (cnt == need || shift == 0) break;  // the whole bucket is taken, or keys are exact
      if (cnt <= 256) {
        resolve = true;
        break;
      }
      hb = shift - 1;
    }
  }
  // bitmaps of the keys above the bucket / in it: four threads per 32-key
  // word (8 keys each), two words per quad per round, OR-combined with two
  // shuffles
  const int W = (n + 31) >> 5;
  const int qd = tid >> 2, sub = tid & 3, wpr = nt >> 1;  // quad, its quarter of a word, words per round
  for (int c0 = 0; c0 < W; c0 += wpr) {  // block-uniform rounds
    uint32_t bg[2] = {0u, 0u}, be[2] = {0u, 0u};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = c0 + 2 * qd + h;
      if (c < W) {
        const int i0 = (c << 5) + 8 * sub;
        if ((c << 5) + 32 <= n16) {
          // chunks 2 sub and 2 sub + 1 of the word, order flipped on odd
          // words: the 8 threads of a quarter-warp hit 8 different bank groups
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int uu = u ^ (c & 1);
            const uint4 v = reinterpret_cast<const uint4*>(keys + i0)[uu];
            const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t xm = x[e] & mask;
              bg[h] |= static_cast<uint32_t>(xm > prefix) << (8 * sub + 4 * uu + e);
              be[h] |= static_cast<uint32_t>(xm == prefix) << (8 * sub + 4 * uu + e);
            }
          }
        } else {
          for (int j = 0; j < 8 && i0 + j < n; ++j) {
            const uint32_t xm = keys[i0 + j] & mask;
            bg[h] |= static_cast<uint32_t>(xm > prefix) << (8 * sub + j);
            be[h] |= static_cast<uint32_t>(xm == prefix) << (8 * sub + j);
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      bg[h] |= __shfl_xor_sync(0xffffffffu, bg[h], 1);
      be[h] |= __shfl_xor_sync(0xffffffffu, be[h], 1);
      bg[h] |= __shfl_xor_sync(0xffffffffu, bg[h], 2);
      be[h] |= __shfl_xor_sync(0xffffffffu, be[h], 2);
      const int c = c0 + 2 * qd + h;
      if (c < W && sub == 0) {
        t.gtw[c] = bg[h];
        t.eqw[c] = be[h];
      }
    }
  }
  if (resolve) {
    // gather the bucket's keys (at most 256) from the non-zero bucket words
    if (tid == 0) t.ncand = 0;
    __syncthreads();
    for (int c0 = 0; c0 < W; c0 += nt) {  // block-uniform rounds (one atomic per warp)
      const int c = c0 + tid;
      const uint32_t be = c < W ? t.eqw[c] : 0u;
      const int m = __popc(be);
      int incl = m;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int wbase = 0;
      if (lane == 31 && incl > 0) wbase = atomicAdd(&t.ncand, incl);
      wbase = __shfl_sync(0xffffffffu, wbase, 31);
      int slot = wbase + incl - m;
      uint32_t e = be;
      while (e) {
        const int j = __ffs(e) - 1;
        e &= e - 1u;
        t.cand[slot] = (c << 5) + j;
        t.candk[slot] = keys[(c << 5) + j];
        ++slot;
      }
    }
  }
  __syncthreads();
  if (resolve) {
    // exact threshold among the bucket's keys (cnt <= 256)
    const int cnt = t.ncand;
    for (int q = tid; q < cnt; q += nt) {
      const uint32_t x = t.candk[q];
      int gt = 0, eq = 0;
#pragma unroll 8
      for (int j = 0; j < cnt; ++j) {
        const uint32_t y = t.candk[j];
        gt += y > x;
        eq += y == x;
      }
      if (gt < need && need <= gt + eq) {  // x is the need-th largest (every such x is equal)
        t.thr = x;
        t.need_thr = need - gt;
      }
    }
    __syncthreads();
    const uint32_t thr = t.thr;
    for (int q = tid; q < cnt; q += nt) {
      const uint32_t x = t.candk[q];
      const int ci = t.cand[q];
      if (x != thr) {
        const uint32_t bit = 1u << (ci & 31);
        if (x > thr) atomicOr(&t.gtw[ci >> 5], bit);
        atomicAnd(&t.eqw[ci >> 5], ~bit);
      }
    }
    need = t.need_thr;
    __syncthreads();
  }
  // words -> ascending indices, thread j owning words [j*wpt, (j+1)*wpt).
  // Keys equal to the threshold are taken in index order, so the number
  // taken before a thread is min(equal keys before it, need).  One block
  // scan carries both counts (equal keys in the high half, keys above in the
  // low half: each total is at most n < 65536).
  {
    const int wpt = (W + nt - 1) / nt;
    const int c0 = min(W, tid * wpt), c1 = min(W, c0 + wpt);
    int e_loc = 0, g_loc = 0;
    for (int c = c0; c < c1; ++c) {
      e_loc += __popc(t.eqw[c]);
      g_loc += __popc(t.gtw[c]);
    }
    const uint32_t packed = block_exclusive_scan_t<uint32_t>(
        (static_cast<uint32_t>(e_loc) << 16) | static_cast<uint32_t>(g_loc),
        reinterpret_cast<uint32_t*>(t.wa), reinterpret_cast<uint32_t*>(&t.total));
    int e_seen = static_cast<int>(packed >> 16);
    int pos = static_cast<int>(packed & 0xffffu) + min(e_seen, need);
    for (int c = c0; c < c1; ++c) {
      uint32_t e = t.eqw[c];
      const uint32_t g = t.gtw[c];
      const int pe = __popc(e);
      if (e_seen >= need) {
        e = 0u;
      } else if (e_seen + pe > need) {  // keep the lowest need - e_seen set bits
        uint32_t keep = 0u;
        for (int r = need - e_seen; r > 0; --r) {
          keep |= e & (~e + 1u);
          e &= e - 1u;
        }
        e = keep;
      }
      e_seen += pe;
      uint32_t f = e | g;
      while (f) {
        dst[pos++] = base + (c << 5) + (__ffs(f) - 1);
        f &= f - 1u;
      }
    }
  }
  __syncthreads();
}

// Adaptive budget (SequenceO1 close reading §3.2: keep the leading items
// whose cumulative importance reaches the fraction p of the total; §4.2:
// softmax of the scores, sorted, cumulative sum, at least one kept).  sel[0,
// k_budget) holds the candidates the fixed budget chose (ascending page ids,
// page p's key at keys[p - base]); keys[0, nc) are every candidate's keys.
// Keeps the smallest prefix of the chosen, in (score desc, page asc) order,
// whose weights exp(tau (s - max s)) add up to at least top_p of the weights
// of all nc candidates, and at least min(k_min, k_budget) of them; rewrites
// sel[0, k) ascending and returns k.  Weights and sums in fp32, each sum in a
// fixed order (a thread's run, then a block scan), so the count does not
// depend on timing.  k_budget <= kMaxTopPPages; scratch: kTopPScratchWords
// words of shared memory; s_wi, s_wf: 36 words each; blockDim.x a multiple
// of 32.  Every thread calls it.
constexpr int kTopPScratchWords = 3 * kMaxTopPPages;

template <typename SelT>
__device__ int topp_trim(const uint32_t* keys, int nc, SelT* sel, int k_budget, int base, float tau,
                         float top_p, int k_min, uint32_t* scratch, int* s_wi, float* s_wf) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  if (k_budget <= 0) return 0;
  // p = 1: no proper prefix holds all the mass (every weight is positive),
  // so the whole budget stays; fp32 sums in two orders cannot show that
  // when a few pages dominate, so it is taken from the definition
  if (top_p >= 1.f) return k_budget;
  uint32_t* ck = scratch;                                        // [k_budget] chosen keys
  float* w = reinterpret_cast<float*>(scratch + kMaxTopPPages);  // [k_budget] weights by rank
  int* rk = reinterpret_cast<int*>(scratch + 2 * kMaxTopPPages); // [k_budget] rank of each
  // the largest key (every chosen key set is a top set: it holds the max)
  uint32_t kmx = 0u;
  for (int i = tid; i < k_budget; i += nt) {
    const uint32_t x = keys[static_cast<int>(sel[i]) - base];
    ck[i] = x;
    kmx = max(kmx, x);
  }
  kmx = __reduce_max_sync(0xffffffffu, kmx);
  if (lane == 0) s_wi[warp] = static_cast<int>(kmx);
  __syncthreads();
  uint32_t m = 0u;
  for (int w2 = 0; w2 < nw; ++w2) m = max(m, static_cast<uint32_t>(s_wi[w2]));
  const float smax = key_score(m);
  // total weight of every candidate: a strided run per thread, then a fixed tree
  float z = 0.f;
  for (int i = tid; i < nc; i += nt) z += expf(tau * (key_score(keys[i]) - smax));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  __syncthreads();  // s_wi read above
  if (lane == 0) s_wf[warp] = z;
  // the rank of each chosen key among the chosen (key desc, page asc)
  for (int i = tid; i < k_budget; i += nt) {
    const uint32_t x = ck[i];
    int r = 0;
    for (int j = 0; j < k_budget; ++j) {
      const uint32_t y = ck[j];
      r += (y > x) || (y == x && j < i);
    }
    w[r] = expf(tau * (key_score(x) - smax));
    rk[i] = r;
  }
  __syncthreads();
  float Z = 0.f;
  for (int w2 = 0; w2 < nw; ++w2) Z += s_wf[w2];
  const float thr = top_p * Z;
  __syncthreads();  // every thread has read the warp sums before the scan reuses them
  // prefix sums of the weights in rank order: thread t owns ranks [r0, r1)
  const int per = (k_budget + nt - 1) / nt;
  const int r0 = min(k_budget, tid * per), r1 = min(k_budget, r0 + per);
  float loc = 0.f;
  for (int r = r0; r < r1; ++r) loc += w[r];
  float pre = block_exclusive_scan_t<float>(loc, s_wf, s_wf + 32);
  int below = 0;  // ranks whose running sum (through them) stays under top_p * Z
  for (int r = r0; r < r1; ++r) {
    pre += w[r];
    below += pre < thr;
  }
  const int n_below = block_exclusive_scan(below, s_wi, s_wi + 32) + below;  // inclusive at the last thread
  if (tid == nt - 1) s_wi[33] = n_below;
  __syncthreads();
  const int k_p = min(s_wi[33] + 1, k_budget);
  const int k = min(k_budget, max(k_p, min(k_min, k_budget)));
  // keep the chosen with rank < k, ascending (sel order): one block scan
  SelT keep_id[1];
  for (int i0 = 0; i0 < k_budget; i0 += nt) {  // block-uniform rounds
    const int i = i0 + tid;
    bool keep = false;
    if (i < k_budget) {
      keep = rk[i] < k;
      keep_id[0] = sel[i];
    }
    __syncthreads();  // every entry of this round read before any is moved
    const int before = i0 == 0 ? 0 : s_wi[34];
    const int pos = block_exclusive_scan(keep ? 1 : 0, s_wi, s_wi + 32);
    if (keep) sel[before + pos] = keep_id[0];
    if (tid == nt - 1) s_wi[34] = before + pos + (keep ? 1 : 0);
    __syncthreads();
  }
  return k;
}

using TopkShared = TopkSmem<8192>;
static_assert(alignof(TopkShared) >= 16 && alignof(TopkSmem<kMaxTopkPages>) >= 16,
              "16-byte accesses to the histogram");

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

// acc + the dot product of the 8 int4 codes of w (two's-complement nibbles;
// even-index codes in the low nibbles) with int8 query codes (q_even, q_odd:
// 4 bytes each), except that every code c enters as c + 8: the nibble with
// its top bit flipped is c + 8 in 0..15, an unsigned byte, so a mask, a shift
// and an XOR replace the sign extension.  The caller subtracts
// sketch_query_bias() once per token: the result is then the exact integer
// dot product.
__device__ __forceinline__ int dot_int4x8_biased(uint32_t w, int q_even, int q_odd, int acc) {
  const uint32_t lo = (w & 0x0f0f0f0fu) ^ 0x08080808u;
  const uint32_t hi = ((w >> 4) & 0x0f0f0f0fu) ^ 0x08080808u;
  asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(lo), "r"(q_even));
  asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(hi), "r"(q_odd));
  return acc;
}
// 8 times the sum of the 16 query codes packed in qc[4]: what the +8 of every
// key code adds to a token's biased dot product
__device__ __forceinline__ int sketch_query_bias(const int* qc) {
  int s = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) s = __dp4a(qc[k], 0x01010101, s);
  return 8 * s;
}

__device__ __forceinline__ int pack_i8x4(int a, int b, int c, int d) {
  return (a & 0xff) | ((b & 0xff) << 8) | ((c & 0xff) << 16) | ((d & 0xff) << 24);
}


// Exact int32 dot of one token's 16 int4 key codes (8 bytes) with the int8
// index query (packed for dp4a in qc[4]; bias = sketch_query_bias(qc)):
// QSI step 1, the integer product before any dequantisation.
__device__ __forceinline__ int sketch_token_dot(uint2 w, const int* qc, int bias) {
  const int dot = dot_int4x8_biased(w.x, qc[0], qc[1], -bias);
  return dot_int4x8_biased(w.y, qc[2], qc[3], dot);
}

// Index query of the sketch selector for one kv-head group, by one warp:
// the group mean of the G query rows (summed in head order, then divided by
// G), projected through P (d x 16, staged in shared memory) with one rounded
// product and one rounded add per step in channel order (the rule of the key
// side), and quantised to int8 with scale max|q~| / 127 (1 when zero), round
// half to even.  s_qbar: d floats of shared memory for this warp.  Every lane
// returns the codes packed for dp4a (even 0-6, odd 1-7, even 8-14, odd
// 9-15) and the scale; lanes j < 16 also return code j in *code_j.
template <typename TQ>
__device__ void sketch_index_query_warp(const TQ* qb, int G, int d, const float* s_P, float* s_qbar,
                                        int lane, int (&qc4)[4], float& sq, int* code_j = nullptr) {
  constexpr int DS = 16;
  for (int i = lane; i < d; i += 32) {
    float s = to_f32(qb[i]);
    for (int g = 1; g < G; ++g) s = __fadd_rn(s, to_f32(qb[static_cast<size_t>(g) * d + i]));
    s_qbar[i] = __fdiv_rn(s, static_cast<float>(G));
  }
  __syncwarp();
  float qt = 0.f;
  if (lane < DS) {
    // one output per lane, its sum in channel order; unrolled so that the
    // shared-memory loads run ahead of the chain of rounded adds (d is a
    // multiple of 32)
#pragma unroll 16
    for (int i = 0; i < d; ++i) qt = __fadd_rn(qt, __fmul_rn(s_qbar[i], s_P[i * DS + lane]));
  }
  float am = fabsf(qt);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  sq = am > 0.f ? __fdiv_rn(am, 127.0f) : 1.0f;
  const int qc = max(-127, min(127, static_cast<int>(rintf(__fdiv_rn(qt, sq)))));
  if (code_j) *code_j = qc;
  int c[DS];
#pragma unroll
  for (int j = 0; j < DS; ++j) c[j] = __shfl_sync(0xffffffffu, qc, j);
  qc4[0] = pack_i8x4(c[0], c[2], c[4], c[6]);
  qc4[1] = pack_i8x4(c[1], c[3], c[5], c[7]);
  qc4[2] = pack_i8x4(c[8], c[10], c[12], c[14]);
  qc4[3] = pack_i8x4(c[9], c[11], c[13], c[15]);
  __syncwarp();  // s_qbar may be reused
}

// The same for a whole CTA: P staged into s_P (d*16 floats) by every
// thread, then warp 0 builds the query; leaves the packed codes in s_qc[4]
// and the scale in *s_sq.
template <typename TQ>
__device__ void sketch_index_query(const TQ* qb, int G, int d, const float* proj, float* s_qbar,
                                   float* s_P, int* s_qc, float* s_sq) {
  constexpr int DS = 16;
  for (int i = threadIdx.x; i < d * DS; i += blockDim.x) s_P[i] = proj[i];
  __syncthreads();
  if (threadIdx.x < 32) {
    int qc4[4];
    float sq;
    sketch_index_query_warp<TQ>(qb, G, d, s_P, s_qbar, threadIdx.x, qc4, sq);
    if (threadIdx.x == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) s_qc[k] = qc4[k];
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
  const int bias = sketch_query_bias(qc);
  float zmax = -INFINITY;
  float z[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    z[k] = -INFINITY;
    if (lane + 32 * k < S) {
      z[k] = static_cast<float>(sketch_token_dot(wk[k], qc, bias)) * cz;
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

// Scores of nb <= 4 consecutive sketch blocks of a staged tile (block r at
// tile + r * rb: S tokens x 8 bytes of int4 codes) by one warp, with the
// four blocks' reductions interleaved: z = dot(codes, qc) * cz[r], score =
// max z + ln sum exp(z - max z) over the block's S <= 128 tokens.
__device__ __forceinline__ void sketch_block_scores4(const uint8_t* tile, int rb, int nb, int S,
                                                     const int* qc, const float (&cz)[4],
                                                     float (&score)[4]) {
  const int lane = threadIdx.x & 31;
  constexpr float kL2e = 1.4426950408889634f;
  const int bias = sketch_query_bias(qc);
  float z[4][4], zmax[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    zmax[r] = -INFINITY;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      z[r][k] = -INFINITY;
      if (r < nb && lane + 32 * k < S) {
        const uint2 w = *reinterpret_cast<const uint2*>(tile + r * rb + (lane + 32 * k) * 8);
        z[r][k] = static_cast<float>(sketch_token_dot(w, qc, bias)) * cz[r] * kL2e;  // log2 domain
        zmax[r] = fmaxf(zmax[r], z[r][k]);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int r = 0; r < 4; ++r) zmax[r] = fmaxf(zmax[r], __shfl_xor_sync(0xffffffffu, zmax[r], o));
  float sum[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    sum[r] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (r < nb && lane + 32 * k < S) sum[r] += exp2f(z[r][k] - zmax[r]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int r = 0; r < 4; ++r) sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], o);
#pragma unroll
  for (int r = 0; r < 4; ++r) score[r] = (zmax[r] + log2f(sum[r])) * kLn2;
}

// Score of one full sketch block (S tokens x 8 bytes of int4 codes at blk)
// for one lane: z_t = dot(codes_t, qc) * cz, score = max z + ln sum exp(z -
// max z), without any exchange between lanes, so that a warp scores up to 32
// blocks at once (lane r taking block r).  Lane r reads token (t + r) mod S
// at step t: the eight-byte reads of a half-warp then fall in different bank
// pairs.  cz > 0 (a product of positive scales), so the maximum logit is cz
// times the maximum integer dot, exactly; a second pass sums exp2 in the log2
// domain.  SC: the block size as a compile-time constant (16, 32 or 64):
// each token's integer dot is then computed once and kept in registers for
// the second pass; 0: any S <= 128 (power of two), dots computed twice.
template <int SC>
__device__ __forceinline__ float sketch_block_score_lane_t(const uint8_t* blk, int S_, const int* qc,
                                                           int bias, float cz) {
  constexpr float kL2e = 1.4426950408889634f;
  const int S = SC > 0 ? SC : S_;
  const int rot = threadIdx.x & (S - 1);
  if constexpr (SC > 0) {
    int d[SC];
    int dmax = INT_MIN;
#pragma unroll
    for (int t = 0; t < SC; ++t) {
      const int tt = (t + rot) & (SC - 1);
      const uint2 w = *reinterpret_cast<const uint2*>(blk + tt * 8);
      d[t] = sketch_token_dot(w, qc, bias);
      dmax = max(dmax, d[t]);
    }
    const float zmax = static_cast<float>(dmax) * cz * kL2e;
    float sum = 0.f;
#pragma unroll
    for (int t = 0; t < SC; ++t) sum += exp2f(static_cast<float>(d[t]) * cz * kL2e - zmax);
    return (zmax + log2f(sum)) * kLn2;
  } else {
    int dmax = INT_MIN;
    for (int t = 0; t < S; ++t) {
      const int tt = (t + rot) & (S - 1);
      const uint2 w = *reinterpret_cast<const uint2*>(blk + tt * 8);
      dmax = max(dmax, sketch_token_dot(w, qc, bias));
    }
    const float zmax = static_cast<float>(dmax) * cz * kL2e;
    float sum = 0.f;
    for (int t = 0; t < S; ++t) {
      const int tt = (t + rot) & (S - 1);
      const uint2 w = *reinterpret_cast<const uint2*>(blk + tt * 8);
      sum += exp2f(static_cast<float>(sketch_token_dot(w, qc, bias)) * cz * kL2e - zmax);
    }
    return (zmax + log2f(sum)) * kLn2;
  }
}

// S: a power of two, 16 <= S <= 128 (warp-uniform)
__device__ __forceinline__ float sketch_block_score_lane(const uint8_t* blk, int S, const int* qc,
                                                         int bias, float cz) {
  if (S == 64) return sketch_block_score_lane_t<64>(blk, S, qc, bias, cz);
  if (S == 32) return sketch_block_score_lane_t<32>(blk, S, qc, bias, cz);
  if (S == 16) return sketch_block_score_lane_t<16>(blk, S, qc, bias, cz);
  return sketch_block_score_lane_t<0>(blk, S, qc, bias, cz);
}

}  // namespace spg
