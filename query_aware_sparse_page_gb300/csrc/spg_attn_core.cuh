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

template <typename T, int D, int G, int NW = kConsumerWarps>
struct AttnConsumer {
  static constexpr int CW = NW;  // warps sharing one staged page
  static constexpr int LPT = G >= 4 ? 16 : 8;  // lanes per token
  static constexpr int TPR = 32 / LPT;         // tokens per warp per round
  static constexpr int RT = CW * TPR;          // tokens per round of the whole stage
  using LC = LaneChannels<T, D, LPT>;
  static constexpr int CPL = LC::CPL;

  float qf[G][CPL], acc[G][CPL], m[G], l[G];
  int cw, tg, lt;

  // qrows: the group's G query rows of D elements (global); scale folded in.
  // cw_: this warp's consumer index (its merge slot); its share of each page
  // is cw_ % NW.
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
        const int t = r0 + rr * RT + (cw % NW) * TPR + tg;
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
          const int t = r0 + rr * RT + (cw % NW) * TPR + tg;
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

// ---- tensor-core consumer ------------------------------------------------------
// Flash-decoding of one staged page on the tensor cores (mma.sync m16n8k16,
// fp32 accumulate) for fp16/bf16 pools, one warp per page.  The group's G
// query rows are the N = 8 columns (zero-padded), tokens and channels the M
// side, so the accumulators are small:
//   S^T [16 tokens x 8 rows]    = K [16 x D] . Q^T [D x 8]       (A = K tile)
//   O^T [D x 8 rows]           += V^T [D x 16 tokens] . P^T [16 x 8]
// K and V come from ldmatrix (V transposed on load); P^T is rounded to the
// pool's 16-bit type as a hi + lo pair (two products, ~16 significant bits
// or more) and moved into the B layout with movmatrix.  The staged page is
// D / 64 tiles of [S rows][64 channels] each for K, then the same for V, as
// the TMA tile copy with 128-byte swizzle leaves them: the 16-byte chunk c of
// row r sits at chunk c ^ (r % 8) of the row (tiles 1024-byte aligned).
//
// Lane layout (g = lane / 4, t = lane % 4): the lane owns query rows 2t and
// 2t + 1: its running max m[e] and sum l[e], and accumulator columns e of
// channels 16 mt + g and 16 mt + g + 8.
template <typename T, int D, int G>
struct AttnMma {
  static_assert(D % 64 == 0, "64-channel tiles");
  static constexpr int KS = D / 16;  // k-steps of Q K^T, m-tiles of P V
  uint32_t qb[KS][2];
  float acc[KS][4];
  float m[2], l[2];
  float scale;
  int cw;

  template <typename TQ>
  __device__ void init(const TQ* qrows, float scale_log2, int cw_, int lane) {
    static_assert(sizeof(TQ) == sizeof(T) && !is_i8<T>(), "same 16-bit type for q and K/V");
    cw = cw_;
    scale = scale_log2;
    const int n = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < KS; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t w = 0;
        if (n < G) {
          const int k = 16 * j + 2 * t + 8 * hf;
          w = *reinterpret_cast<const uint32_t*>(qrows + n * D + k);
        }
        qb[j][hf] = w;
      }
#pragma unroll
    for (int j = 0; j < KS; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }

  // one staged page (shared memory, 1024-byte aligned) with nv valid tokens
  // (0 < nv <= S, S a multiple of 16); the slots past nv are zeroed first
  // when the page is the sequence's last, partial one
  __device__ void consume(uint8_t* st, int S, int nv, int lane) {
    constexpr int NH = D / 64;
    const uint32_t kb = smem_u32(st);
    const uint32_t vb = kb + static_cast<uint32_t>(S) * D * sizeof(T);
    const uint32_t hs = static_cast<uint32_t>(S) * 128u;  // bytes of one 64-channel tile
    if (nv < S) {
      // rows past the end hold whatever the pool holds: make them zeros so
      // that p = 0 times them stays 0 in the P V product
      const int words = (S - nv) * NH * 8;
      for (int i = lane; i < words; i += 32) {
        const int r = nv + i / (NH * 8), rem = i % (NH * 8);
        *reinterpret_cast<uint4*>(st + S * D * sizeof(T) + (rem >> 3) * hs + r * 128 + (rem & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }
    const int g = lane >> 2, mi = lane >> 3, r8 = lane & 7;
    for (int t0 = 0; t0 < nv; t0 += 16) {
      // S^T tile: two accumulation chains over the k-steps
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int tok = t0 + (mi & 1) * 8 + r8;  // A rows: tokens
        const uint32_t rowb = kb + tok * 128u;
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          const int chunk = 2 * j + (mi >> 1);
          uint32_t a[4];
          ldmatrix_x4(a, rowb + (chunk >> 3) * hs + (((chunk & 7) ^ (tok & 7)) << 4));
          if (j & 1)
            mma_16816<T>(c1, a, qb[j][0], qb[j][1]);
          else
            mma_16816<T>(c0, a, qb[j][0], qb[j][1]);
        }
      }
      float sv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sv[e] = (c0[e] + c1[e]) * scale;
      if (t0 + 16 > nv) {
        if (t0 + g >= nv) sv[0] = sv[1] = -INFINITY;
        if (t0 + g + 8 >= nv) sv[2] = sv[3] = -INFINITY;
      }
      // running max of rows 2t, 2t+1 over this tile's tokens (lanes with equal t)
      float mx0 = fmaxf(sv[0], sv[2]), mx1 = fmaxf(sv[1], sv[3]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      if (mx0 > m[0]) {
        const float corr = exp2f(m[0] - mx0);
        m[0] = mx0;
        l[0] *= corr;
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          acc[j][0] *= corr;
          acc[j][2] *= corr;
        }
      }
      if (mx1 > m[1]) {
        const float corr = exp2f(m[1] - mx1);
        m[1] = mx1;
        l[1] *= corr;
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          acc[j][1] *= corr;
          acc[j][3] *= corr;
        }
      }
      const float p0 = exp2f(sv[0] - m[0]), p1 = exp2f(sv[1] - m[1]);
      const float p2 = exp2f(sv[2] - m[0]), p3 = exp2f(sv[3] - m[1]);
      l[0] += p0 + p2;
      l[1] += p1 + p3;
      // P^T as B fragments: hi and lo 16-bit parts, tokens 0-7 and 8-15
      const uint32_t h01 = pack2<T>(p0, p1), h23 = pack2<T>(p2, p3);
      const float2 f01 = unpack2f<T>(h01), f23 = unpack2f<T>(h23);
      const uint32_t l01 = pack2<T>(p0 - f01.x, p1 - f01.y), l23 = pack2<T>(p2 - f23.x, p3 - f23.y);
      const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
      const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);
      {
        const int tok = t0 + (mi >> 1) * 8 + r8;  // stored rows of the transposed loads
        const uint32_t rowb = vb + tok * 128u;
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          const int chunk = 2 * j + (mi & 1);
          uint32_t a[4];
          ldmatrix_x4_trans(a, rowb + (chunk >> 3) * hs + (((chunk & 7) ^ (tok & 7)) << 4));
          mma_16816<T>(acc[j], a, bh0, bh1);
          mma_16816<T>(acc[j], a, bl0, bl1);
        }
      }
    }
  }

  // the sums of rows 2t, 2t+1 over the warp's lanes (the max is already uniform)
  __device__ void fold() {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], o);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], o);
    }
  }

  // this warp's state into s_m/s_l [CW][G] and s_acc [CW][G][D]
  __device__ void store(float* s_m, float* s_l, float* s_acc, int lane) const {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int row = 2 * t + e;
      if (row < G) {
        if (g == 0) {
          s_m[cw * G + row] = m[e];
          s_l[cw * G + row] = l[e];
        }
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          s_acc[(cw * G + row) * D + 16 * j + g] = acc[j][e];
          s_acc[(cw * G + row) * D + 16 * j + g + 8] = acc[j][e + 2];
        }
      }
    }
  }
};

// ---- tensor-core consumer for int8 pools ---------------------------------------
// The same flash-decoding step for int8 K/V with fp16 per-token scales (SALS
// SFAA: antiquant attention), fp16 query, D = 128.  int8 codes become fp16
// exactly in registers: the byte biased to unsigned (x ^ 0x80) is placed
// under an fp16 exponent byte 0x64 (the value 1024 + x + 128) and 1152 is
// subtracted.  The staged page is the K tile [S rows][128 bytes] and the V
// tile, each as left by a TMA tile copy with 128-byte swizzle (chunk c of row
// r at chunk c ^ (r % 8)), then the S fp16 K scales and S fp16 V scales.
//   S^T = K Q^T: ldmatrix on the int8 rows read as 16-bit pairs gives a lane
//     4 consecutive channels 4q..4q+3 of one token (q = lane % 4) of a
//     16-channel chunk; the k index of the mma is mapped to channels
//     (2q, 2q+1 -> 4q, 4q+1; 2q+8, 2q+9 -> 4q+2, 4q+3), and the query's B
//     fragments use the same map.  The logit of token t is multiplied by its
//     K scale.
//   O^T += V^T P'^T with p' = 256 p * (V scale of the token) (the power of
//     two keeps small p' out of fp16's subnormal range; undone at the store):
//     ldmatrix.trans on
//     16-bit pairs gives a lane tokens (2q, 2q+1) x channels (2g, 2g+1); the
//     m-tile's rows g and g + 8 are mapped to channels 2g and 2g + 1 of the
//     chunk.
template <int G>
struct AttnMmaI8 {
  static constexpr int D = 128;
  static constexpr int NC = D / 16;  // 16-channel chunks: k-steps of Q K^T, m-tiles of P V
  uint32_t qb[NC][2];
  float acc[NC][4];
  float m[2], l[2];
  float scale;
  int cw;

  // the lane's four consecutive int8 channels -> fp16 pairs (bytes 0,1 / 2,3)
  __device__ static __forceinline__ void i8x4_to_h2(uint32_t r, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = r ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    const __half2 bias = __floats2half2_rn(1152.f, 1152.f);
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<const uint32_t*>(&ha);
    hi = *reinterpret_cast<const uint32_t*>(&hb);
  }
  // bytes (0, 2) and (1, 3) of a transposed load -> fp16 pairs
  __device__ static __forceinline__ void i8x4t_to_h2(uint32_t r, uint32_t& e, uint32_t& o) {
    const uint32_t u = r ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4240;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4341;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    const __half2 bias = __floats2half2_rn(1152.f, 1152.f);
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    e = *reinterpret_cast<const uint32_t*>(&ha);
    o = *reinterpret_cast<const uint32_t*>(&hb);
  }

  __device__ void init(const __half* qrows, float scale_log2, int cw_, int lane) {
    cw = cw_;
    scale = scale_log2;
    const int n = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < NC; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        // k = 2t (+8 hf), 2t + 1 (+8 hf) -> channels 16 j + 4 t + 2 hf, + 1
        uint32_t w = 0;
        if (n < G) w = *reinterpret_cast<const uint32_t*>(qrows + n * D + 16 * j + 4 * t + 2 * hf);
        qb[j][hf] = w;
      }
#pragma unroll
    for (int j = 0; j < NC; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }

  // S^T of the 16 tokens at t0 (K codes at kb) against the query: the
  // lane's logits sv (tokens t0 + g, t0 + g + 8; query columns 2t, 2t + 1),
  // scaled by the tokens' K scales and the softmax scale, -inf past nv
  __device__ __forceinline__ void qk16(uint32_t kb, const __half* ksc, int S, int nv, int t0,
                                       int lane, float (&sv)[4]) const {
    const int g = lane >> 2, mi = lane >> 3, r8 = lane & 7;
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    const int tok = t0 + (mi & 1) * 8 + r8;
    const uint32_t rowb = kb + tok * D;
#pragma unroll
    for (int j = 0; j < NC; j += 2) {
      const int chunk = j + (mi >> 1);
      uint32_t r[4];
      ldmatrix_x4(r, rowb + ((chunk ^ (tok & 7)) << 4));
      // r[0]: tokens 0-7 of chunk j, r[1]: tokens 8-15, r[2], r[3]: chunk j + 1
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t a[4];
        i8x4_to_h2(r[2 * h], a[0], a[2]);
        i8x4_to_h2(r[2 * h + 1], a[1], a[3]);
        if (h == 0)
          mma_16816<__half>(c0, a, qb[j][0], qb[j][1]);
        else
          mma_16816<__half>(c1, a, qb[j + 1][0], qb[j + 1][1]);
      }
    }
    const float ks0 = __half2float(ksc[min(t0 + g, S - 1)]);
    const float ks1 = __half2float(ksc[min(t0 + g + 8, S - 1)]);
    sv[0] = (c0[0] + c1[0]) * ks0 * scale;
    sv[1] = (c0[1] + c1[1]) * ks0 * scale;
    sv[2] = (c0[2] + c1[2]) * ks1 * scale;
    sv[3] = (c0[3] + c1[3]) * ks1 * scale;
    if (t0 + g >= nv) sv[0] = sv[1] = -INFINITY;
    if (t0 + g + 8 >= nv) sv[2] = sv[3] = -INFINITY;
  }

  // O^T += V^T P^T for the 16 tokens at t0 (V codes at vb), p the lane's
  // probabilities of those tokens (layout of qk16's sv)
  __device__ __forceinline__ void pv16(uint32_t vb, const __half* vsc, int nv, int t0, int lane,
                                       const float (&p)[4]) {
    const int g = lane >> 2, r8 = lane & 7;
    // p' = 256 p * V scale of the token (0 past the end)
    const float vs0 = t0 + g < nv ? 256.f * __half2float(vsc[t0 + g]) : 0.f;
    const float vs1 = t0 + g + 8 < nv ? 256.f * __half2float(vsc[t0 + g + 8]) : 0.f;
    const float q0 = p[0] * vs0, q1 = p[1] * vs0, q2 = p[2] * vs1, q3 = p[3] * vs1;
    const uint32_t h01 = pack2<__half>(q0, q1), h23 = pack2<__half>(q2, q3);
    const float2 f01 = unpack2f<__half>(h01), f23 = unpack2f<__half>(h23);
    const uint32_t l01 = pack2<__half>(q0 - f01.x, q1 - f01.y);
    const uint32_t l23 = pack2<__half>(q2 - f23.x, q3 - f23.y);
    const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
    const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);
    // matrices: tokens 0-7 / 8-15 of chunk j (lanes 0-15), then of chunk j + 1
    const int tok = t0 + ((lane >> 3) & 1) * 8 + r8;
    const uint32_t rowb = vb + tok * D;
#pragma unroll
    for (int j = 0; j < NC; j += 2) {
      const int chunk = j + (lane >> 4);
      uint32_t r[4];
      ldmatrix_x4_trans(r, rowb + ((chunk ^ (tok & 7)) << 4));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t a[4];
        i8x4t_to_h2(r[2 * h], a[0], a[1]);      // tokens 0-7: rows g (ch 2g), g + 8 (ch 2g + 1)
        i8x4t_to_h2(r[2 * h + 1], a[2], a[3]);  // tokens 8-15
        mma_16816<__half>(acc[j + h], a, bh0, bh1);
        mma_16816<__half>(acc[j + h], a, bl0, bl1);
      }
    }
  }

  // one staged page with nv valid tokens (0 < nv <= S, S a multiple of 16),
  // 32 tokens per step: the two 16-token products are independent, and one
  // online-softmax update (max, rescale, exp) serves both
  __device__ void consume(uint8_t* st, int S, int nv, int lane) {
    const uint32_t kb = smem_u32(st);
    const uint32_t vb = kb + static_cast<uint32_t>(S) * D;
    const __half* ksc = reinterpret_cast<const __half*>(st + 2 * S * D);
    const __half* vsc = ksc + S;
    if (nv < S) {
      // V rows past the end: zeros (their p' is 0, but 0 times a stale value
      // could be NaN inside the product)
      const int words = (S - nv) * 8;
      for (int i = lane; i < words; i += 32)
        *reinterpret_cast<uint4*>(st + S * D + (nv + i / 8) * D + (i % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
      __syncwarp();
    }
    for (int t0 = 0; t0 < nv; t0 += 32) {
      const bool two = t0 + 16 < nv;  // the second 16 tokens hold a valid one
      float sa[4], sb[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      qk16(kb, ksc, S, nv, t0, lane, sa);
      if (two) qk16(kb, ksc, S, nv, t0 + 16, lane, sb);
      float mx0 = fmaxf(fmaxf(sa[0], sa[2]), fmaxf(sb[0], sb[2]));
      float mx1 = fmaxf(fmaxf(sa[1], sa[3]), fmaxf(sb[1], sb[3]));
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      if (mx0 > m[0]) {
        const float corr = exp2f(m[0] - mx0);
        m[0] = mx0;
        l[0] *= corr;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          acc[j][0] *= corr;
          acc[j][2] *= corr;
        }
      }
      if (mx1 > m[1]) {
        const float corr = exp2f(m[1] - mx1);
        m[1] = mx1;
        l[1] *= corr;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          acc[j][1] *= corr;
          acc[j][3] *= corr;
        }
      }
      float pa[4], pb[4];
      pa[0] = exp2f(sa[0] - m[0]);
      pa[1] = exp2f(sa[1] - m[1]);
      pa[2] = exp2f(sa[2] - m[0]);
      pa[3] = exp2f(sa[3] - m[1]);
      pb[0] = exp2f(sb[0] - m[0]);
      pb[1] = exp2f(sb[1] - m[1]);
      pb[2] = exp2f(sb[2] - m[0]);
      pb[3] = exp2f(sb[3] - m[1]);
      l[0] += (pa[0] + pa[2]) + (pb[0] + pb[2]);
      l[1] += (pa[1] + pa[3]) + (pb[1] + pb[3]);
      pv16(vb, vsc, nv, t0, lane, pa);
      if (two) pv16(vb, vsc, nv, t0 + 16, lane, pb);
    }
  }

  __device__ void fold() {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], o);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], o);
    }
  }

  // rows g / g + 8 of m-tile j hold channels 16 j + 2 g / 16 j + 2 g + 1
  __device__ void store(float* s_m, float* s_l, float* s_acc, int lane) const {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int row = 2 * t + e;
      if (row < G) {
        if (g == 0) {
          s_m[cw * G + row] = m[e];
          s_l[cw * G + row] = l[e];
        }
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          s_acc[(cw * G + row) * D + 16 * j + 2 * g] = acc[j][e] * (1.f / 256.f);
          s_acc[(cw * G + row) * D + 16 * j + 2 * g + 1] = acc[j][e + 2] * (1.f / 256.f);
        }
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
