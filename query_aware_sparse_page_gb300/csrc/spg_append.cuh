// Metadata append of the token just written at position L - 1 of a
// sequence, shared by the single-launch decode kernels.
//
// Quest 完全拆解, 关键性估计算法: the page's per-channel minimum and maximum
// are updated with the new key (the page's first token starts them afresh).
// SALS长序列推理优化, the low-rank index key: when the token completes a
// block, the block's keys are dequantised, projected through P and quantised
// to int4 with one scale per block.
#pragma once

#include "spg_attn_core.cuh"
#include "spg_common.cuh"

namespace spg {

// Quest append of token L-1 of (b, h) by one warp.  minmax is the
// [B][Hkv][MP][2][D] logical-page metadata with chunk-swizzled rows.
template <typename T, int D>
__device__ void minmax_append_warp(const T* k_pool, const int32_t* page_table, T* minmax,
                                   int32_t* err, int Hkv, int S, int MP, int n_phys, int b, int h,
                                   int L, int lane) {
  constexpr int CPL = D / 32;
  const int t = L - 1, p = t / S, slot = t % S;
  const int phys = page_table[static_cast<size_t>(b) * MP + p];
  if (phys < 0 || phys >= n_phys) {
    if (lane == 0) record_error(err, SPG_DEVERR_PAGE_ID);
    return;
  }
  const size_t ph = static_cast<size_t>(phys) * Hkv + h;
  const T* k = k_pool + (ph * S + slot) * D + lane * CPL;
  T* row = minmax + ((static_cast<size_t>(b) * Hkv + h) * MP + p) * 2 * D;
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const T kv = k[c];
    T& lo = row[meta_swz<T>(lane * CPL + c, p)];
    T& hi = row[meta_swz<T>(D + lane * CPL + c, p)];
    if (slot == 0) {
      lo = kv;
      hi = kv;
    } else {
      const float kf = to_f32(kv);
      if (kf < to_f32(lo)) lo = kv;
      if (kf > to_f32(hi)) hi = kv;
    }
  }
}

// fp32 -> 16-bit type rounded toward -inf / +inf (the Quest interval of
// int8 keys is stored rounded outward, so it still holds every key)
template <typename TM> __device__ __forceinline__ TM round_down16(float x);
template <typename TM> __device__ __forceinline__ TM round_up16(float x);
template <> __device__ __forceinline__ __half round_down16<__half>(float x) { return __float2half_rd(x); }
template <> __device__ __forceinline__ __half round_up16<__half>(float x) { return __float2half_ru(x); }
template <> __device__ __forceinline__ __nv_bfloat16 round_down16<__nv_bfloat16>(float x) {
  return __float2bfloat16_rd(x);
}
template <> __device__ __forceinline__ __nv_bfloat16 round_up16<__nv_bfloat16>(float x) {
  return __float2bfloat16_ru(x);
}

// Quest append of token L-1 of (b, h) over an int8 pool with per-token fp16
// scales (Quest 完全拆解, 与量化的兼容性: the metadata taken from the
// quantised keys): the dequantised key code * scale (exact in fp32) widens
// the page's interval, stored in TM rounded outward.  One warp.
template <typename TM, int D>
__device__ void minmax_append_warp_i8(const int8_t* k_pool, const __half* k_scale,
                                      const int32_t* page_table, TM* minmax, int32_t* err, int Hkv,
                                      int S, int MP, int n_phys, int b, int h, int L, int lane) {
  constexpr int CPL = D / 32;
  const int t = L - 1, p = t / S, slot = t % S;
  const int phys = page_table[static_cast<size_t>(b) * MP + p];
  if (phys < 0 || phys >= n_phys) {
    if (lane == 0) record_error(err, SPG_DEVERR_PAGE_ID);
    return;
  }
  const size_t ph = static_cast<size_t>(phys) * Hkv + h;
  const int8_t* k = k_pool + (ph * S + slot) * D + lane * CPL;
  const float sc = __half2float(k_scale[ph * S + slot]);
  TM* row = minmax + ((static_cast<size_t>(b) * Hkv + h) * MP + p) * 2 * D;
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const float v = __fmul_rn(static_cast<float>(k[c]), sc);
    const TM dn = round_down16<TM>(v), up = round_up16<TM>(v);
    TM& lo = row[meta_swz<TM>(lane * CPL + c, p)];
    TM& hi = row[meta_swz<TM>(D + lane * CPL + c, p)];
    if (slot == 0) {
      lo = dn;
      hi = up;
    } else {
      if (to_f32(dn) < to_f32(lo)) lo = dn;
      if (to_f32(up) > to_f32(hi)) hi = up;
    }
  }
}

// 16 consecutive channels of a key row as fp32 (row 16-byte aligned)
template <typename T>
__device__ __forceinline__ void load16_f32(const T* p, float (&x)[16]) {
  if constexpr (sizeof(T) == 1) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 16; ++e) x[e] = static_cast<float>(static_cast<int8_t>((ws[e >> 2] >> (8 * (e & 3))) & 0xffu));
  } else {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) load_cvt<T, 8>(p + 8 * hf, x + 8 * hf);
  }
}

// The 16 projected values of one key row: deq(k) . P with each product
// rounded and the sum taken in channel order (no fused multiply-add); int8
// keys are dequantised by their fp16 scale first (exact in fp32).
template <typename T, int D>
__device__ __forceinline__ void sketch_project_row(const T* krow, float sc, const float* proj,
                                                   float (&v)[16]) {
  constexpr int DS = 16;
#pragma unroll
  for (int u = 0; u < DS; ++u) v[u] = 0.f;
  const float4* P4 = reinterpret_cast<const float4*>(proj);  // [D][DS] row-major
  for (int ic = 0; ic < D; ic += 16) {
    float x[16];
    load16_f32<T>(krow + ic, x);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float kv = x[e];
      if constexpr (is_i8<T>()) kv = __fmul_rn(kv, sc);
#pragma unroll
      for (int q4 = 0; q4 < DS / 4; ++q4) {
        const float4 pv = __ldg(P4 + (ic + e) * (DS / 4) + q4);
        v[4 * q4] = __fadd_rn(v[4 * q4], __fmul_rn(kv, pv.x));
        v[4 * q4 + 1] = __fadd_rn(v[4 * q4 + 1], __fmul_rn(kv, pv.y));
        v[4 * q4 + 2] = __fadd_rn(v[4 * q4 + 2], __fmul_rn(kv, pv.z));
        v[4 * q4 + 3] = __fadd_rn(v[4 * q4 + 3], __fmul_rn(kv, pv.w));
      }
    }
  }
}

// The projected values of one key row for the sketch outputs [u0, u0 + NU)
// (u0 a multiple of 4), in the same order as sketch_project_row (each
// product rounded, each output's sum in channel order): splitting the 16
// outputs between lanes gives the same values.
template <typename T, int D, int NU>
__device__ __forceinline__ void sketch_project_row_part(const T* krow, float sc, const float* proj,
                                                        int u0, float (&v)[NU]) {
  constexpr int DS = 16;
#pragma unroll
  for (int u = 0; u < NU; ++u) v[u] = 0.f;
  const float4* P4 = reinterpret_cast<const float4*>(proj) + u0 / 4;  // [D][DS] row-major
  for (int ic = 0; ic < D; ic += 16) {
    float x[16];
    load16_f32<T>(krow + ic, x);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float kv = x[e];
      if constexpr (is_i8<T>()) kv = __fmul_rn(kv, sc);
#pragma unroll
      for (int q4 = 0; q4 < NU / 4; ++q4) {
        const float4 pv = __ldg(P4 + (ic + e) * (DS / 4) + q4);
        v[4 * q4] = __fadd_rn(v[4 * q4], __fmul_rn(kv, pv.x));
        v[4 * q4 + 1] = __fadd_rn(v[4 * q4 + 1], __fmul_rn(kv, pv.y));
        v[4 * q4 + 2] = __fadd_rn(v[4 * q4 + 2], __fmul_rn(kv, pv.z));
        v[4 * q4 + 3] = __fadd_rn(v[4 * q4 + 3], __fmul_rn(kv, pv.w));
      }
    }
  }
}

// Sketch of block blk of (b, h) by a whole CTA (blockDim.x >= S): thread t
// projects token t, the block scale is absmax / 7 (1 for an all-zero
// block), codes rint(v / scale) clamped to [-7, 7], two per byte, channel
// 2j in the low nibble.  s_red: blockDim.x / 32 floats of shared memory.
// Every thread of the CTA calls it.
template <typename T, int D>
__device__ void sketch_block_cta(const T* k_pool, const __half* k_scale, const int32_t* page_table,
                                 const float* proj, uint8_t* sketch, float* sketch_scale,
                                 int32_t* err, int Hkv, int S, int MP, int n_phys, int b, int h,
                                 int blk, float* s_red) {
  constexpr int DS = 16;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int phys = page_table[static_cast<size_t>(b) * MP + blk];
  const bool ok = phys >= 0 && phys < n_phys;
  if (!ok && tid == 0) record_error(err, SPG_DEVERR_PAGE_ID);
  float v[DS];
  float amax = 0.f;
#pragma unroll
  for (int u = 0; u < DS; ++u) v[u] = 0.f;
  if (ok && tid < S) {
    const size_t ph = static_cast<size_t>(phys) * Hkv + h;
    float sc = 1.f;
    if constexpr (is_i8<T>()) sc = __half2float(k_scale[ph * S + tid]);
    sketch_project_row<T, D>(k_pool + (ph * S + tid) * D, sc, proj, v);
#pragma unroll
    for (int u = 0; u < DS; ++u) amax = fmaxf(amax, fabsf(v[u]));
  }
  amax = warp_max(amax);
  if (lane == 0) s_red[warp] = amax;
  __syncthreads();
  amax = 0.f;
  for (int w = 0; w < nw; ++w) amax = fmaxf(amax, s_red[w]);
  __syncthreads();  // s_red may be reused by the caller
  if (!ok) return;
  const float scale = amax > 0.f ? __fdiv_rn(amax, 7.0f) : 1.0f;
  const size_t lrow = (static_cast<size_t>(b) * Hkv + h) * MP + blk;
  if (tid < S) {
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < DS / 2; ++k) {
      const int c0 = max(-7, min(7, static_cast<int>(rintf(__fdiv_rn(v[2 * k], scale)))));
      const int c1 = max(-7, min(7, static_cast<int>(rintf(__fdiv_rn(v[2 * k + 1], scale)))));
      w[k >> 2] |= static_cast<uint32_t>((c0 & 0xf) | ((c1 & 0xf) << 4)) << (8 * (k & 3));
    }
    *reinterpret_cast<uint2*>(sketch + (lrow * S + tid) * (DS / 2)) = make_uint2(w[0], w[1]);
  }
  if (tid == 0) sketch_scale[lrow] = scale;
}

}  // namespace spg
