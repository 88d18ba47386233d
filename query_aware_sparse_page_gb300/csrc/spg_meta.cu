// Page metadata maintenance.
//
// Quest (Quest 完全拆解, 关键性估计算法): per page and kv-head, the per-channel
// min m and max M of the page's keys, updated by one compare per channel when
// a token is inserted.  The page's first token starts the statistics afresh,
// so pages can be recycled without clearing.
//
// Metadata is stored per sequence in logical page order ([B][Hkv][MP][...]),
// not per physical page: the scan of one (sequence, kv-head) then reads one
// contiguous range, in large bulk copies, and needs no page-table lookup.
// Quest rows are chunk-swizzled by page (meta_swz).
//
// Sketch (SALS长序列推理优化, 算法简介 "low rank 预处理" and QSI's int4 index
// key): when a block of S tokens is complete, its keys are dequantised,
// projected through the fixed d x ds matrix P (fp32, one rounded product and
// one rounded add per step, channels in order: the codes are defined by this
// arithmetic) and quantised to int4 in [-7, 7] with one scale max|k~|/7.
// The open tail block is never scored, so it is quantised only once full.
#include "spg_append.cuh"
#include "spg_common.cuh"
#include "spg_internal.h"

namespace spg {
namespace {

// CPL consecutive elements moved as one 4- or 8-byte word
template <typename T, int CPL>
struct alignas(CPL * sizeof(T)) Vec {
  T v[CPL];
};

// Append, Quest: one warp per (batch, kv-head); each lane owns CPL
// consecutive channels of the new key and of the page's m and M rows.
template <typename T, int CPL>
__global__ void k_minmax_append(const T* __restrict__ k_pool, const int32_t* __restrict__ page_table,
                                const int32_t* __restrict__ seq_lens, T* __restrict__ minmax,
                                int B, int Hkv, int S, int d, int MP, int n_phys,
                                int32_t* __restrict__ err) {
  pdl_wait();
  pdl_trigger();
  const int unit = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (unit >= B * Hkv) return;
  const int b = unit / Hkv, h = unit % Hkv;
  const int L = seq_lens[b];
  if (L <= 0) {
    if (L < 0 && lane == 0) record_error(err, SPG_DEVERR_SEQ_LEN);
    return;
  }
  if (L > MP * S) {
    if (lane == 0) record_error(err, SPG_DEVERR_SEQ_LEN);
    return;
  }
  const int t = L - 1, p = t / S, slot = t % S;
  const int phys = page_table[(size_t)b * MP + p];
  if (phys < 0 || phys >= n_phys) {
    if (lane == 0) record_error(err, SPG_DEVERR_PAGE_ID);
    return;
  }
  using V = Vec<T, CPL>;
  const V k = *reinterpret_cast<const V*>(k_pool + (((size_t)phys * Hkv + h) * S + slot) * d +
                                          lane * CPL);
  const size_t mrow = ((size_t)unit * MP + p) * 2 * d;  // [B][Hkv][MP][2][d]
  V* lo = reinterpret_cast<V*>(minmax + mrow + meta_swz<T>(lane * CPL, p));
  V* hi = reinterpret_cast<V*>(minmax + mrow + meta_swz<T>(d + lane * CPL, p));
  if (slot == 0) {  // the page's first token starts its statistics
    *lo = k;
    *hi = k;
    return;
  }
  V m = *lo, M = *hi;
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const float kf = to_f32(k.v[c]);
    if (kf < to_f32(m.v[c])) m.v[c] = k.v[c];
    if (kf > to_f32(M.v[c])) M.v[c] = k.v[c];
  }
  *lo = m;
  *hi = M;
}

// Rebuild, Quest: one warp per (batch, kv-head, page).
template <typename T>
__global__ void k_minmax_rebuild(const T* __restrict__ k_pool, const int32_t* __restrict__ page_table,
                                 const int32_t* __restrict__ seq_lens, T* __restrict__ minmax,
                                 int B, int Hkv, int S, int d, int MP, int n_phys,
                                 int32_t* __restrict__ err) {
  const int warps_per_block = blockDim.x >> 5;
  const int p = blockIdx.x * warps_per_block + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int unit = blockIdx.y;
  const int b = unit / Hkv, h = unit % Hkv;
  const int L = seq_lens[b];
  if (L < 0 || L > MP * S) {
    if (p == 0 && lane == 0) record_error(err, SPG_DEVERR_SEQ_LEN);
    return;
  }
  const int P = (L + S - 1) / S;
  if (p >= P) return;
  const int phys = page_table[(size_t)b * MP + p];
  if (phys < 0 || phys >= n_phys) {
    if (lane == 0) record_error(err, SPG_DEVERR_PAGE_ID);
    return;
  }
  const int n_valid = min(S, L - p * S);
  const T* base = k_pool + ((size_t)phys * Hkv + h) * S * d;
  T* mrow = minmax + ((size_t)unit * MP + p) * 2 * d;  // [B][Hkv][MP][2][d]
  for (int c = lane; c < d; c += 32) {
    T lo = base[c], hi = base[c];
    float lof = to_f32(lo), hif = lof;
    for (int t = 1; t < n_valid; ++t) {
      const T k = base[(size_t)t * d + c];
      const float kf = to_f32(k);
      if (kf < lof) { lo = k; lof = kf; }
      if (kf > hif) { hi = k; hif = kf; }
    }
    mrow[meta_swz<T>(c, p)] = lo;
    mrow[meta_swz<T>(d + c, p)] = hi;
  }
}

// Quest over int8 keys with per-token fp16 scales (Quest 完全拆解,
// 与量化的兼容性): the interval of the dequantised keys code * scale (exact in
// fp32), stored in the query's 16-bit type TM rounded outward.
// Append: one warp per (batch, kv-head).
template <typename TM, int D>
__global__ void k_minmax_append_i8(const int8_t* __restrict__ k_pool, const __half* __restrict__ k_scale,
                                   const int32_t* __restrict__ page_table,
                                   const int32_t* __restrict__ seq_lens, TM* __restrict__ minmax,
                                   int B, int Hkv, int S, int MP, int n_phys, int32_t* __restrict__ err) {
  pdl_wait();
  pdl_trigger();
  const int unit = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (unit >= B * Hkv) return;
  const int b = unit / Hkv, h = unit % Hkv;
  const int L = seq_lens[b];
  if (L <= 0 || L > MP * S) {
    if (L != 0 && lane == 0) record_error(err, SPG_DEVERR_SEQ_LEN);
    return;
  }
  minmax_append_warp_i8<TM, D>(k_pool, k_scale, page_table, minmax, err, Hkv, S, MP, n_phys, b, h, L,
                               lane);
}

// Rebuild: one warp per (batch, kv-head, page); fp32 min / max over the
// page's valid tokens, then one outward rounding each.
template <typename TM>
__global__ void k_minmax_rebuild_i8(const int8_t* __restrict__ k_pool, const __half* __restrict__ k_scale,
                                    const int32_t* __restrict__ page_table,
                                    const int32_t* __restrict__ seq_lens, TM* __restrict__ minmax,
                                    int B, int Hkv, int S, int d, int MP, int n_phys,
                                    int32_t* __restrict__ err) {
  const int warps_per_block = blockDim.x >> 5;
  const int p = blockIdx.x * warps_per_block + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int unit = blockIdx.y;
  const int b = unit / Hkv, h = unit % Hkv;
  const int L = seq_lens[b];
  if (L < 0 || L > MP * S) {
    if (p == 0 && lane == 0) record_error(err, SPG_DEVERR_SEQ_LEN);
    return;
  }
  const int P = (L + S - 1) / S;
  if (p >= P) return;
  const int phys = page_table[(size_t)b * MP + p];
  if (phys < 0 || phys >= n_phys) {
    if (lane == 0) record_error(err, SPG_DEVERR_PAGE_ID);
    return;
  }
  const int n_valid = min(S, L - p * S);
  const size_t ph = (size_t)phys * Hkv + h;
  const int8_t* base = k_pool + ph * S * d;
  const __half* sc = k_scale + ph * S;
  TM* mrow = minmax + ((size_t)unit * MP + p) * 2 * d;  // [B][Hkv][MP][2][d]
  for (int c = lane; c < d; c += 32) {
    float lo = INFINITY, hi = -INFINITY;
    for (int t = 0; t < n_valid; ++t) {
      const float v = __fmul_rn(static_cast<float>(base[(size_t)t * d + c]), __half2float(sc[t]));
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
    mrow[meta_swz<TM>(c, p)] = round_down16<TM>(lo);
    mrow[meta_swz<TM>(d + c, p)] = round_up16<TM>(hi);
  }
}

template <typename TM>
cudaError_t meta_quest_i8(const spg_params& p, const void* k_pool, const void* k_scale,
                          const int32_t* pt, const int32_t* lens, int rebuild, void* minmax,
                          int32_t* err, cudaStream_t st) {
  const int B = p.batch, Hkv = p.num_kv_heads, S = p.page_size, d = p.head_dim;
  const int MP = p.max_pages_per_seq, NP = p.num_phys_pages;
  const int8_t* kp = static_cast<const int8_t*>(k_pool);
  const __half* ks = static_cast<const __half*>(k_scale);
  TM* mm = static_cast<TM*>(minmax);
  if (!rebuild) {
    const int threads = 128, units = B * Hkv;
    const int blocks = (units * 32 + threads - 1) / threads;
    if (d == 128)
      return launch_pdl(k_minmax_append_i8<TM, 128>, dim3(blocks), dim3(threads), 0, st, kp, ks, pt,
                        lens, mm, B, Hkv, S, MP, NP, err);
    return launch_pdl(k_minmax_append_i8<TM, 64>, dim3(blocks), dim3(threads), 0, st, kp, ks, pt, lens,
                      mm, B, Hkv, S, MP, NP, err);
  }
  const int wpb = 8;
  dim3 grid((MP + wpb - 1) / wpb, B * Hkv);
  k_minmax_rebuild_i8<TM><<<grid, wpb * 32, 0, st>>>(kp, ks, pt, lens, mm, B, Hkv, S, d, MP, NP, err);
  return cudaGetLastError();
}

template <typename T>
__device__ __forceinline__ float dequant_key(const T* row, const __half* scale, int i) {
  return to_f32(row[i]);
}
template <>
__device__ __forceinline__ float dequant_key<int8_t>(const int8_t* row, const __half* scale, int i) {
  // int8 code x fp16 scale: both exact in fp32, and so is their product
  return __fmul_rn(static_cast<float>(row[i]), __half2float(*scale));
}

// Sketch of one full block: CTA per (block, batch*kv-head).  append != 0 ->
// only the block completed by the token at seq_len-1.
template <typename T>
__global__ void k_sketch_block(const T* __restrict__ k_pool, const __half* __restrict__ k_scale,
                               const int32_t* __restrict__ page_table,
                               const int32_t* __restrict__ seq_lens, const float* __restrict__ proj,
                               uint8_t* __restrict__ sketch, float* __restrict__ sketch_scale,
                               int B, int Hkv, int S, int d, int ds, int MP, int n_phys,
                               int append, int32_t* __restrict__ err) {
  extern __shared__ __align__(16) float sm[];
  float* sP = sm;                  // [d][ds]
  float* sK = sP + d * ds;         // [S][d]  dequantised keys
  float* sV = sK + S * d;          // [S][ds] projected keys
  __shared__ float s_red[32];

  const int unit = blockIdx.y;
  const int b = unit / Hkv, h = unit % Hkv;
  const int L = seq_lens[b];
  if (L < 0 || L > MP * S) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_error(err, SPG_DEVERR_SEQ_LEN);
    return;
  }
  int blk;
  if (append) {
    if (L == 0 || (L % S) != 0) return;  // no block completed by this token
    blk = L / S - 1;
  } else {
    blk = blockIdx.x;
    if ((blk + 1) * S > L) return;  // only full blocks
  }
  const int phys = page_table[(size_t)b * MP + blk];
  if (phys < 0 || phys >= n_phys) {
    if (threadIdx.x == 0) record_error(err, SPG_DEVERR_PAGE_ID);
    return;
  }
  const size_t ph = (size_t)phys * Hkv + h;
  const T* kb = k_pool + ph * S * d;
  for (int i = threadIdx.x; i < d * ds; i += blockDim.x) sP[i] = proj[i];
  for (int i = threadIdx.x; i < S * d; i += blockDim.x) {
    const int t = i / d, c = i % d;
    const __half* sc = k_scale ? k_scale + ph * S + t : nullptr;
    sK[i] = dequant_key<T>(kb + (size_t)t * d, sc, c);
  }
  __syncthreads();

  // k~[t][j] = sum_i k[t][i] * P[i][j]: sequential in i, unfused
  float amax = 0.f;
  for (int o = threadIdx.x; o < S * ds; o += blockDim.x) {
    const int t = o / ds, j = o % ds;
    float acc = 0.f;
    for (int i = 0; i < d; ++i) acc = __fadd_rn(acc, __fmul_rn(sK[t * d + i], sP[i * ds + j]));
    sV[o] = acc;
    amax = fmaxf(amax, fabsf(acc));
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? s_red[threadIdx.x] : 0.f;
    v = warp_max(v);
    if (threadIdx.x == 0) s_red[0] = v;
  }
  __syncthreads();
  const float a = s_red[0];
  const float scale = a > 0.f ? __fdiv_rn(a, 7.0f) : 1.0f;

  // codes, two per byte (channel 2j in the low nibble)
  const size_t lrow = (size_t)unit * MP + blk;  // [B][Hkv][MP] logical block
  uint8_t* out = sketch + lrow * S * (ds / 2);
  for (int o2 = threadIdx.x; o2 < S * ds / 2; o2 += blockDim.x) {
    const float v0 = sV[2 * o2], v1 = sV[2 * o2 + 1];
    int c0 = static_cast<int>(rintf(__fdiv_rn(v0, scale)));
    int c1 = static_cast<int>(rintf(__fdiv_rn(v1, scale)));
    c0 = max(-7, min(7, c0));
    c1 = max(-7, min(7, c1));
    out[o2] = static_cast<uint8_t>((c0 & 0xf) | ((c1 & 0xf) << 4));
  }
  if (threadIdx.x == 0) sketch_scale[lrow] = scale;
}

template <typename T>
cudaError_t meta_typed(const spg_params& p, const void* k_pool, const void* k_scale,
                       const int32_t* pt, const int32_t* lens, int rebuild, void* minmax,
                       uint8_t* sketch, float* sketch_scale, const float* proj, int32_t* err,
                       cudaStream_t st) {
  const int B = p.batch, Hkv = p.num_kv_heads, S = p.page_size, d = p.head_dim;
  const int MP = p.max_pages_per_seq, NP = p.num_phys_pages;
  const T* kp = static_cast<const T*>(k_pool);
  if (p.selector == SPG_SEL_QUEST && is_i8<T>()) {
    return p.q_dtype == SPG_F16
               ? meta_quest_i8<__half>(p, k_pool, k_scale, pt, lens, rebuild, minmax, err, st)
               : meta_quest_i8<__nv_bfloat16>(p, k_pool, k_scale, pt, lens, rebuild, minmax, err, st);
  }
  if (p.selector == SPG_SEL_QUEST) {
    if (!rebuild) {
      const int threads = 128, units = B * Hkv;
      const int blocks = (units * 32 + threads - 1) / threads;
      T* mm = static_cast<T*>(minmax);
      if (d == 128)
        return launch_pdl(k_minmax_append<T, 4>, dim3(blocks), dim3(threads), 0, st, kp, pt, lens,
                          mm, B, Hkv, S, d, MP, NP, err);
      return launch_pdl(k_minmax_append<T, 2>, dim3(blocks), dim3(threads), 0, st, kp, pt, lens,
                        mm, B, Hkv, S, d, MP, NP, err);
    } else {
      const int wpb = 8;
      dim3 grid((MP + wpb - 1) / wpb, B * Hkv);
      k_minmax_rebuild<T><<<grid, wpb * 32, 0, st>>>(kp, pt, lens, static_cast<T*>(minmax), B,
                                                     Hkv, S, d, MP, NP, err);
    }
  } else if (p.selector == SPG_SEL_SKETCH_INT4) {
    const int ds = p.sketch_dim;
    const size_t smem = sizeof(float) * ((size_t)d * ds + (size_t)S * d + (size_t)S * ds);
    auto kern = k_sketch_block<T>;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
      if (e != cudaSuccess) return e;
    }
    dim3 grid(rebuild ? MP : 1, B * Hkv);
    kern<<<grid, 256, smem, st>>>(kp, static_cast<const __half*>(k_scale), pt, lens, proj, sketch,
                                  sketch_scale, B, Hkv, S, d, ds, MP, NP, rebuild ? 0 : 1, err);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_meta_update(const spg_params& p, const void* k_pool, const void* k_scale,
                               const int32_t* page_table, const int32_t* seq_lens, int rebuild,
                               void* minmax, uint8_t* sketch, float* sketch_scale,
                               const float* proj, int32_t* err, cudaStream_t stream) {
  switch (p.kv_dtype) {
    case SPG_F16:
      return meta_typed<__half>(p, k_pool, k_scale, page_table, seq_lens, rebuild, minmax, sketch,
                                sketch_scale, proj, err, stream);
    case SPG_BF16:
      return meta_typed<__nv_bfloat16>(p, k_pool, k_scale, page_table, seq_lens, rebuild, minmax,
                                       sketch, sketch_scale, proj, err, stream);
    default:
      return meta_typed<int8_t>(p, k_pool, k_scale, page_table, seq_lens, rebuild, minmax, sketch,
                                sketch_scale, proj, err, stream);
  }
}

}  // namespace spg
