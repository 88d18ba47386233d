// The consumer side of flash-decoding over one staged KV page, shared by the
// split-K attention kernel and the fused single-launch decode step.
//
// Sources: SALS长序列推理优化, SFAA (QK^T, online softmax, P@V, rescale; int8
// K/V dequantised by their per-token scales); Quest 完全拆解, Approximate
// attention.
//
// A stage holds one page of one kv-head: K [S][D], V [S][D] and, for int8
// pools, the fp16 K scales [S] and V scales [S].  kConsumerWarps warps share
// it: each takes TPR tokens of every RT-token round, LPT lanes per token (8,
// or 16 when the group has 4 or 8 query rows, to bound registers).  A lane's
// channels are 16-byte chunks lt, lt + LPT, ... of the row (or one smaller
// piece), so the lanes of a token hit distinct bank groups and each shared
// load runs at the minimum number of wavefronts.  Logits of the G query rows
// reduce over the token's lanes with shuffles; the running max per row is
// warp-wide, the accumulator per lane covers the lane's channels of its
// token group, and token groups are folded once at the end.
#pragma once

#include "spg_common.cuh"

namespace spg {

constexpr int kConsumerWarps = 4;
constexpr int kMaxStages = 8;

template <typename T>
__host__ __device__ constexpr bool is_i8() { return sizeof(T) == 1; }

// bytes of one staged page: K tile, V tile, and for int8 the two fp16 scale rows
template <typename T, int D>
__host__ __device__ inline uint32_t kv_stage_bytes(int S) {
  const uint32_t tile = static_cast<uint32_t>(S) * D * sizeof(T);
  const uint32_t sc = is_i8<T>() ? static_cast<uint32_t>(S) * 2 : 0u;
  return 2 * tile + 2 * sc;
}

// Which channels of a row a lane owns: NLD loads of EPL consecutive elements.
template <typename T, int D, int LPT>
struct LaneChannels {
  static constexpr int CPL = D / LPT;  // channels per lane
  static constexpr int BYTES = CPL * static_cast<int>(sizeof(T));
  static constexpr int NLD = BYTES >= 16 ? BYTES / 16 : 1;  // loads per row
  static constexpr int EPL = CPL / NLD;                     // elements per load
  // first channel of load k for lane-in-token lt
  __device__ static constexpr int base(int lt, int k) {
    return BYTES >= 16 ? (lt + LPT * k) * EPL : lt * CPL;
  }
  __device__ static void load(const T* row, int lt, float* o) {
#pragma unroll
    for (int k = 0; k < NLD; ++k) load_cvt<T, EPL>(row + base(lt, k), o + k * EPL);
  }
};

template <typename T, int D, int G>
struct AttnConsumer {
  static constexpr int CW = kConsumerWarps;
  static constexpr int LPT = G >= 4 ? 16 : 8;  // lanes per token
  static constexpr int TPR = 32 / LPT;         // tokens per warp per round
  static constexpr int RT = CW * TPR;          // tokens per round of the whole stage
  using LC = LaneChannels<T, D, LPT>;
  static constexpr int CPL = LC::CPL;

  float qf[G][CPL], acc[G][CPL], m[G], l[G];
  int cw, tg, lt;

  // qrows: the group's G query rows of D elements (global); scale folded in
  template <typename TQ>
  __device__ void init(const TQ* qrows, float scale_log2, int cw_, int lane) {
    cw = cw_;
    tg = lane / LPT;
    lt = lane % LPT;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int k = 0; k < LC::NLD; ++k)
#pragma unroll
        for (int e = 0; e < LC::EPL; ++e) {
          qf[g][k * LC::EPL + e] = to_f32(qrows[g * D + LC::base(lt, k) + e]) * scale_log2;
          acc[g][k * LC::EPL + e] = 0.f;
        }
    }
  }

  // one staged page with nv valid tokens (0 < nv <= S)
  __device__ void consume(const uint8_t* st, int S, int nv) {
    const uint32_t tile = static_cast<uint32_t>(S) * D * sizeof(T);
    const T* Ks = reinterpret_cast<const T*>(st);
    const T* Vs = reinterpret_cast<const T*>(st + tile);
    const __half* ksc = reinterpret_cast<const __half*>(st + 2 * tile);
    const __half* vsc = ksc + S;
    for (int r0 = 0; r0 < nv; r0 += 4 * RT) {
      // logits of up to 4 rounds of this warp's tokens
      float z[4][G];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int t = r0 + rr * RT + cw * TPR + tg;
#pragma unroll
        for (int g = 0; g < G; ++g) z[rr][g] = -INFINITY;
        if (r0 + rr * RT < nv) {  // warp-uniform
          float kf[CPL];
          const int tr = min(t, S - 1);
          LC::load(Ks + tr * D, lt, kf);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float part = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) part = fmaf(qf[g][c], kf[c], part);
#pragma unroll
            for (int o = 1; o < LPT; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if constexpr (is_i8<T>()) part *= __half2float(ksc[tr]);
            if (t < nv) z[rr][g] = part;
          }
        }
      }
      // warp-wide max of the new logits; rescale only when it grows
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float cm = fmaxf(fmaxf(z[0][g], z[1][g]), fmaxf(z[2][g], z[3][g]));
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        if (cm > m[g]) {
          const float corr = exp2f(m[g] - cm);
          m[g] = cm;
          l[g] *= corr;
#pragma unroll
          for (int c = 0; c < CPL; ++c) acc[g][c] *= corr;
        }
      }
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        if (r0 + rr * RT < nv) {
          const int t = r0 + rr * RT + cw * TPR + tg;
          const int tr = min(t, S - 1);
          float vf[CPL];
          LC::load(Vs + tr * D, lt, vf);
          float vsv = 1.f;
          if constexpr (is_i8<T>()) vsv = __half2float(vsc[tr]);
          if (t < nv) {  // slots past the sequence end hold arbitrary values
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float p = exp2f(z[rr][g] - m[g]);
              l[g] += p;
              const float pv = p * vsv;
#pragma unroll
              for (int c = 0; c < CPL; ++c) acc[g][c] = fmaf(pv, vf[c], acc[g][c]);
            }
          }
        }
      }
    }
  }

  // fold the warp's token groups together (one running max per warp)
  __device__ void fold() {
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int o = LPT; o < 32; o <<= 1) {
        l[g] += __shfl_xor_sync(0xffffffffu, l[g], o);
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[g][c] += __shfl_xor_sync(0xffffffffu, acc[g][c], o);
      }
    }
  }

  // this warp's state into s_m/s_l [CW][G] and s_acc [CW][G][D] (natural channel order)
  __device__ void store(float* s_m, float* s_l, float* s_acc, int lane) const {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (lane == 0) {
        s_m[cw * G + g] = m[g];
        s_l[cw * G + g] = l[g];
      }
      if (tg == 0) {
#pragma unroll
        for (int k = 0; k < LC::NLD; ++k)
#pragma unroll
          for (int e = 0; e < LC::EPL; ++e)
            s_acc[(cw * G + g) * D + LC::base(lt, k) + e] = acc[g][k * LC::EPL + e];
      }
    }
  }
};

// Log-sum-exp merge of n states (m, l, acc) for one (row g, channel c):
// m_i in the log2 domain; returns the merged max, sum and accumulator.
__device__ __forceinline__ void lse_merge(const float* s_m, const float* s_l, const float* s_acc,
                                          int n, int G, int D, int g, int c, float& M, float& Ls,
                                          float& A) {
  M = -INFINITY;
  for (int w = 0; w < n; ++w) M = fmaxf(M, s_m[w * G + g]);
  A = 0.f;
  Ls = 0.f;
  if (M == -INFINITY) return;
  for (int w = 0; w < n; ++w) {
    const float f = exp2f(s_m[w * G + g] - M);
    A = fmaf(s_acc[(w * G + g) * D + c], f, A);
    Ls = fmaf(s_l[w * G + g], f, Ls);
  }
}

}  // namespace spg
