// sparse_decode_attention_noalloc: the sparse attention entry point for
// callers that cannot allocate device memory.
//
// Some callers of this library have no way to obtain device memory at the
// point where they run decode attention: plugins inside a host framework
// that owns every device allocation and hands its plugins no allocator and
// no workspace, or latency-critical serving loops whose rules forbid
// cudaMalloc (it can stall the whole device) once the model is loaded.  They
// still own q, the pools, the page table and the outputs, but not a
// workspace.  This entry point gives them the split-K attention with its
// scratch (the split partials and an error word) in one fixed array of
// device memory that belongs to the library.
//
// The array is a file-scope __device__ variable of SPG_NOALLOC_SCRATCH_BYTES
// bytes: every GPU that loads the library holds it until the process exits.
// Host code cannot use the variable's name as a device address, so the
// first call on each device (with that device current) looks the address up
// with cudaGetSymbolAddress and caches it; make that first call before any
// stream capture.  Every call on a device shares the one array and leaves
// its contents behind, so calls whose kernels overlap on the GPU (different
// streams, no ordering between them) race and corrupt each other's results.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "spg_common.cuh"
#include "spg_internal.h"

namespace {

constexpr size_t kScratchBytes = SPG_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// bytes of scratch one call needs: error word header, split arrival
// counters, split partials
size_t scratch_needed(const spg_params& p) {
  const size_t rows = static_cast<size_t>(p.batch) * p.num_q_heads;
  const size_t units = static_cast<size_t>(p.batch) * p.num_kv_heads;
  return 256 + round256(sizeof(int32_t) * units) +
         2 * round256(sizeof(float) * rows * spg::kMaxSplits) +
         round256(sizeof(float) * rows * spg::kMaxSplits * p.head_dim);
}

spg_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPG_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return SPG_ECUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return SPG_OK;
}

bool ok16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" spg_status sparse_decode_attention_noalloc(
    const spg_params* p, const void* q, const void* k_pool, const void* v_pool,
    const void* k_scale, const void* v_scale, const int32_t* page_table, const int32_t* seq_lens,
    const int32_t* sel, const int32_t* sel_cnt, float* out, float* lse, spg_stream_t stream) {
  spg_status s = spg_validate(p);
  if (s != SPG_OK) return s;
  if (p->selector == SPG_SEL_ALL) return SPG_EINVAL;
  if (!ok16(q) || !ok16(k_pool) || !ok16(v_pool) || !ok16(page_table) || !ok16(seq_lens) ||
      !ok16(sel) || !ok16(sel_cnt) || !ok16(out) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 15u)))
    return SPG_EINVAL;
  if (p->kv_dtype == SPG_I8 && (!ok16(k_scale) || !ok16(v_scale))) return SPG_EINVAL;
  if (scratch_needed(*p) > kScratchBytes) return SPG_EWORKSPACE;

  void* base = nullptr;
  if ((s = scratch_address(&base)) != SPG_OK) return s;
  const size_t rows = static_cast<size_t>(p->batch) * p->num_q_heads;
  uint8_t* b = static_cast<uint8_t*>(base);
  spg::Workspace w{};
  w.err = reinterpret_cast<int32_t*>(b);
  w.scores = nullptr;  // attention does not score pages
  size_t off = 256;
  const size_t units = static_cast<size_t>(p->batch) * p->num_kv_heads;
  w.counters = reinterpret_cast<int32_t*>(b + off);
  off += round256(sizeof(int32_t) * units);
  w.pm = reinterpret_cast<float*>(b + off);
  off += round256(sizeof(float) * rows * spg::kMaxSplits);
  w.pl = reinterpret_cast<float*>(b + off);
  off += round256(sizeof(float) * rows * spg::kMaxSplits);
  w.pacc = reinterpret_cast<float*>(b + off);

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the error word and the split arrival counters are read before they are
  // written: start them at zero (header and counters are contiguous)
  if (cudaMemsetAsync(b, 0, 256 + round256(sizeof(int32_t) * units), st) != cudaSuccess)
    return SPG_ECUDA;
  const cudaError_t e = spg::launch_attention(*p, q, k_pool, v_pool, k_scale, v_scale, page_table,
                                              seq_lens, sel, sel_cnt, out, lse, w, st);
  return e == cudaSuccess ? SPG_OK : SPG_ECUDA;
}
