// Device helpers shared by the sparse-page kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>
#include <utility>

#include "spg.h"

namespace spg {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxSplits = 128;  // split-K partials per (batch, q-head) held in the workspace
constexpr int kMaxTopkPages = 49152;  // candidate keys of one (batch, kv-head) kept in shared memory
constexpr int kMaxTopPPages = 1024;   // largest page budget of the adaptive (top-p) selection
constexpr int kDefaultProbes = 8;     // probe selector: sampled tokens per page when n_probe is 0

// ---- element conversions -------------------------------------------------
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(int8_t x) { return static_cast<float>(x); }

// 4 consecutive elements of a row -> fp32 (the row pointer is 4-element aligned)
template <typename T>
__device__ __forceinline__ void load4_f32(const T* p, float* o);

template <>
__device__ __forceinline__ void load4_f32<__half>(const __half* p, float* o) {
  uint2 r = *reinterpret_cast<const uint2*>(p);
  float2 a = __half22float2(*reinterpret_cast<__half2*>(&r.x));
  float2 b = __half22float2(*reinterpret_cast<__half2*>(&r.y));
  o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
}
template <>
__device__ __forceinline__ void load4_f32<__nv_bfloat16>(const __nv_bfloat16* p, float* o) {
  uint2 r = *reinterpret_cast<const uint2*>(p);
  // bf16 -> fp32 is a 16-bit shift of the bit pattern
  o[0] = __uint_as_float(r.x << 16);
  o[1] = __uint_as_float(r.x & 0xffff0000u);
  o[2] = __uint_as_float(r.y << 16);
  o[3] = __uint_as_float(r.y & 0xffff0000u);
}
template <>
__device__ __forceinline__ void load4_f32<int8_t>(const int8_t* p, float* o) {
  uint32_t r = *reinterpret_cast<const uint32_t*>(p);
  o[0] = static_cast<float>(static_cast<int8_t>(r & 0xff));
  o[1] = static_cast<float>(static_cast<int8_t>((r >> 8) & 0xff));
  o[2] = static_cast<float>(static_cast<int8_t>((r >> 16) & 0xff));
  o[3] = static_cast<float>(static_cast<int8_t>(r >> 24));
}

// N consecutive elements (N * sizeof(T) in {4, 8, 16} bytes, aligned) -> fp32
template <typename T, int N>
__device__ __forceinline__ void load_cvt(const T* p, float* o) {
  constexpr int BYTES = N * static_cast<int>(sizeof(T));
  static_assert(BYTES == 4 || BYTES == 8 || BYTES == 16, "4, 8 or 16 bytes");
  uint32_t w[BYTES / 4];
  if constexpr (BYTES == 16) {
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
  } else if constexpr (BYTES == 8) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    w[0] = r.x; w[1] = r.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
#pragma unroll
  for (int i = 0; i < BYTES / 4; ++i) {
    if constexpr (sizeof(T) == 1) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[4 * i + j] = static_cast<float>(static_cast<int8_t>((w[i] >> (8 * j)) & 0xffu));
    } else if constexpr (std::is_same<T, __half>::value) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      o[2 * i] = f.x;
      o[2 * i + 1] = f.y;
    } else {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

// 2 consecutive elements -> fp32
template <typename T>
__device__ __forceinline__ void load2_f32(const T* p, float* o) {
  o[0] = to_f32(p[0]);
  o[1] = to_f32(p[1]);
}

__device__ __forceinline__ void record_error(int32_t* err, int32_t bit) {
  if (err) atomicOr(err, bit);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---- shared-memory barriers and bulk async copies (TMA bulk engine) -------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// make barrier initialisation visible to the async proxy before first use
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// kCluster: acquire at cluster scope (the phase was completed by arrivals
// from other CTAs of the cluster, see mbar_arrive_cluster)
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (kCluster)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  return ok != 0;
}

// arrive on the mbarrier at shared::cluster address `addr` (another CTA's),
// release at cluster scope: what this thread did before (and what a CTA
// barrier ordered before that) is visible to a cluster-scope wait that sees
// the phase complete
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// arrive on the mbarrier at shared::cluster address `addr` (another CTA's)
// and add `bytes` to its expected transaction count.  Relaxed: it orders
// nothing before it (a release would first wait for this thread's earlier
// global stores); the data it waits for come with st_async_u32.
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(addr),
               "r"(bytes)
               : "memory");
}

// asynchronous 32-bit store into another CTA's shared memory: `addr` and the
// mbarrier `bar` are shared::cluster addresses in that CTA; the store's
// arrival completes 4 bytes of the barrier's transaction count
__device__ __forceinline__ void st_async_u32(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(addr),
               "r"(v), "r"(bar)
               : "memory");
}

// Bounded wait: returns false when the barrier phase did not complete within
// `limit` polls or 100 ms of wall time, whichever comes first (the caller
// records SPG_DEVERR_TIMEOUT and stops issuing).
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t limit = (1u << 22)) {
  if (mbar_try_wait<kCluster>(bar, parity)) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t i = 1; i < limit; ++i) {
    if (mbar_try_wait<kCluster>(bar, parity)) return true;
    if ((i & 255u) == 0) {
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > 100ull * 1000 * 1000) return false;
    }
  }
  return false;
}

// global -> shared bulk copy; dst, src 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// same, with an L2 evict-first hint: streamed KV pages are read once per step
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// adds `bytes` to the transaction count the barrier's current phase waits for
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// ---- tensor-core fragments (mma.sync m16n8k16, fp32 accumulate) -------------
// ldmatrix: lane i gives the address of row i % 8 of 8x8 matrix i / 8 (16
// bytes); register j holds matrix j in the mma fragment layout (thread t: row
// t / 4, columns 2 (t % 4) and 2 (t % 4) + 1).  The .trans form delivers each
// matrix transposed (thread t: column t / 4, rows 2 (t % 4), 2 (t % 4) + 1).
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// transpose of an 8x8 16-bit matrix held in the fragment layout
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// D = A B + D, A 16x16 (row), B 16x8 (col), fp16 or bf16 operands
template <typename T>
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  if constexpr (std::is_same<T, __half>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// two floats -> packed pair of T (round to nearest), first in the low half
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (std::is_same<T, __half>::value) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}
// the packed pair back to fp32
template <typename T>
__device__ __forceinline__ float2 unpack2f(uint32_t w) {
  if constexpr (std::is_same<T, __half>::value) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  } else {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
}

// ---- TMA tensor tiles ---------------------------------------------------------
// 2-D tile of a tensor map (x: innermost element coordinate, a multiple of 16
// bytes; y: row) into shared memory, completing on `bar`, with an L2 policy.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// brings [p, p + bytes) into L2 (bytes a multiple of 16, p 16-byte aligned)
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- thread-block clusters and distributed shared memory ---------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster; orders shared-memory accesses
// (local and remote) before it with those after it
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// The same barrier split in two, for a cluster's first phase: every thread
// arrives (relaxed) as soon as it starts, and waits before its first access
// to another CTA's shared memory, so that every CTA of the cluster has
// started by then.  Every thread of every CTA calls each once, in this order,
// before its next cluster barrier.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// shared::cluster address of `p` (a shared variable) in CTA `rank`
__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// ---- programmatic dependent launch ------------------------------------------
// Kernels are launched with programmatic stream serialisation: a kernel may be
// scheduled while its predecessor drains, runs its prologue, and waits here
// before it reads anything a predecessor may have written.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// lets the next kernel in the stream start its prologue
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Raises a kernel's dynamic shared-memory limit when its static plus dynamic
// shared memory exceeds the default 48 KB.  The attribute belongs to the
// current device, so the cache of what was raised is keyed by (device,
// kernel) and guarded by a lock: host threads may launch concurrently and
// one thread may drive several GPUs.  Repeated calls are no-ops.
template <typename... KArgs>
inline cudaError_t ensure_smem(void (*kern)(KArgs...), size_t bytes) {
  struct Entry {
    int dev;
    const void* fn;
    size_t bytes;
  };
  static Entry cache[256];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const void* fn = reinterpret_cast<const void*>(kern);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].dev == dev && cache[i].fn == fn && cache[i].bytes >= bytes) return cudaSuccess;
  cudaFuncAttributes attr{};
  e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.sharedSizeBytes + bytes > 48 * 1024)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  int i = 0;
  while (i < n && !(cache[i].dev == dev && cache[i].fn == fn)) ++i;
  if (i < n) {
    cache[i].bytes = bytes > cache[i].bytes ? bytes : cache[i].bytes;
  } else if (n < 256) {
    cache[n++] = Entry{dev, fn, bytes};
  }
  return cudaSuccess;
}

// Quest metadata row layout: a row holds m (d channels) then M (d channels)
// of one (sequence, kv-head, logical page); its 16-byte chunks are stored
// XOR-swizzled by the page index, chunk j at j ^ (p % 8), so that 8
// consecutive pages read at the same logical chunk hit 8 different bank
// groups (conflict-free ldmatrix on a staged tile).  Element offset of
// channel e (0 <= e < 2d) of page p's row:
template <typename T>
__host__ __device__ __forceinline__ int meta_swz(int e, int p) {
  constexpr int EPC = 16 / static_cast<int>(sizeof(T));
  return ((e / EPC) ^ (p & 7)) * EPC + (e % EPC);
}

// the score of a key (inverse of score_key)
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// order-preserving map of an fp32 score to uint32 (larger float -> larger key);
// -0 is first turned into +0 (-0 + +0 = +0 when rounding to nearest), so that
// the two zeros, equal as values, get one key and tie by page index
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(__fadd_rn(s, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace spg
