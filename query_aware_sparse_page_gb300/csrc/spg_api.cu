// C ABI of libspg: parameter validation, workspace layout, launch sequencing.
// Everything here runs on the host; all device work is in the kernel files.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "spg_common.cuh"
#include "spg_internal.h"

namespace spg {

int n_sel_pages(const spg_params& p) { return p.token_budget / p.page_size; }

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < 64) cached[dev] = n;
  return n;
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace layout (every region 256-byte aligned):
//   header    256 B: error word at 0, the scheduled step's queue counters at
//             64, the bounded-wait test hook at 128
//   counters  [B*Hkv] int32: split arrivals of the attention kernel
//   sel_cnt.  [B*Hkv] int32: scoring CTAs done, for the fused selection
//   scores    [B*Hkv][MP] fp32 (the scheduled step keeps its keys here)
//   pm, pl    [B*Hq][kMaxSplits] fp32; pacc [B*Hq][kMaxSplits][d] fp32
//   flags     [4][B*Hkv] int32 (scheduled step)
//   slices    [B*Hkv][n_sel] int2 (scheduled step)
//   iq        [B*Hkv][8] int32 (scheduled step, sketch selector)
size_t workspace_bytes(const spg_params& p) {
  const size_t B = p.batch, Hq = p.num_q_heads, Hkv = p.num_kv_heads;
  const size_t d = p.head_dim, MP = p.max_pages_per_seq;
  const size_t n_sel = p.selector == SPG_SEL_ALL ? 1 : std::max(1, n_sel_pages(p));
  size_t off = 256;                                      // header: error word, queue counters
  off += align256(sizeof(int32_t) * B * Hkv);            // split arrival counters
  off += align256(sizeof(int32_t) * B * Hkv);            // scoring arrival counters
  off += align256(sizeof(float) * B * Hkv * MP);         // scores / keys
  off += align256(sizeof(float) * B * Hq * kMaxSplits);  // pm
  off += align256(sizeof(float) * B * Hq * kMaxSplits);  // pl
  off += align256(sizeof(float) * B * Hq * kMaxSplits * d);  // pacc
  off += align256(sizeof(int32_t) * 4 * B * Hkv);        // per-unit flags
  off += align256(sizeof(int2) * B * Hkv * n_sel);       // selection slices
  off += align256(sizeof(int32_t) * 8 * B * Hkv);        // index queries
  return off;
}

Workspace carve_workspace(const spg_params& p, void* ws) {
  const size_t B = p.batch, Hq = p.num_q_heads, Hkv = p.num_kv_heads, d = p.head_dim;
  const size_t MP = p.max_pages_per_seq;
  const size_t n_sel = p.selector == SPG_SEL_ALL ? 1 : std::max(1, n_sel_pages(p));
  uint8_t* base = static_cast<uint8_t*>(ws);
  Workspace w{};
  w.err = reinterpret_cast<int32_t*>(base);
  w.sched_ctr = reinterpret_cast<int32_t*>(base + 64);
  w.hook = reinterpret_cast<int32_t*>(base + 128);
  size_t off = 256;
  w.counters = reinterpret_cast<int32_t*>(base + off);
  off += align256(sizeof(int32_t) * B * Hkv);
  w.sel_counters = reinterpret_cast<int32_t*>(base + off);
  off += align256(sizeof(int32_t) * B * Hkv);
  w.scores = reinterpret_cast<float*>(base + off);
  off += align256(sizeof(float) * B * Hkv * MP);
  w.pm = reinterpret_cast<float*>(base + off);
  off += align256(sizeof(float) * B * Hq * kMaxSplits);
  w.pl = reinterpret_cast<float*>(base + off);
  off += align256(sizeof(float) * B * Hq * kMaxSplits);
  w.pacc = reinterpret_cast<float*>(base + off);
  off += align256(sizeof(float) * B * Hq * kMaxSplits * d);
  w.sched_flags = reinterpret_cast<int32_t*>(base + off);
  off += align256(sizeof(int32_t) * 4 * B * Hkv);
  w.slices = reinterpret_cast<int2*>(base + off);
  off += align256(sizeof(int2) * B * Hkv * n_sel);
  w.iq = reinterpret_cast<int32_t*>(base + off);
  return w;
}

}  // namespace spg

using spg::Workspace;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }

spg_status check_ws(const spg_params* p, const void* ws, size_t ws_bytes) {
  if (!ok_ptr(ws)) return SPG_EINVAL;
  if (ws_bytes < spg::workspace_bytes(*p)) return SPG_EWORKSPACE;
  return SPG_OK;
}

spg_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SPG_OK : SPG_ECUDA; }

// the selector's metadata inputs
spg_status check_meta_inputs(const spg_params* p, const void* minmax, const uint8_t* sketch,
                             const float* sketch_scale, const float* proj) {
  // (the probe selector's "metadata" is the K pool itself)
  if (p->selector == SPG_SEL_QUEST || p->selector == SPG_SEL_PROBE)
    return ok_ptr(minmax) ? SPG_OK : SPG_EINVAL;
  if (p->selector == SPG_SEL_SKETCH_INT4)
    return (ok_ptr(sketch) && ok_ptr(sketch_scale) && ok_ptr(proj)) ? SPG_OK : SPG_EINVAL;
  return SPG_EINVAL;  // SPG_SEL_ALL has no metadata and no selection
}

// Kernel preference for the single-launch step, process-wide
// (spg_set_step_kernel): 0 automatic, 1 cluster kernel, 2 scheduled kernel.
std::atomic<int> g_step_pref{0};

bool use_fused(const spg_params& p, int append) {
  return g_step_pref.load() != 2 && spg::fused_supported(p, append);
}
bool use_sched(const spg_params& p, int append) {
  return g_step_pref.load() != 1 && spg::sched_supported(p, append);
}

// select + attend: one cluster launch when the parameters allow it (the
// faster single-launch kernel on every measured workload), else one
// persistent scheduled launch, else the scoring/selection launch followed by
// the split-K attention launch.  With append != 0 the single-launch kernels
// also apply the metadata append of the new token.
cudaError_t select_attend(const spg_params& p, const void* q, const void* k_pool,
                          const void* v_pool, const void* k_scale, const void* v_scale,
                          const int32_t* page_table, const int32_t* seq_lens, void* minmax,
                          const uint8_t* sketch, const float* sketch_scale, const float* proj,
                          int32_t* sel, int32_t* sel_cnt, float* out, float* lse, int append,
                          const Workspace& w, cudaStream_t st) {
  if (use_fused(p, append)) {
    const cudaError_t e = spg::launch_fused(p, q, k_pool, v_pool, k_scale, v_scale, page_table,
                                            seq_lens, minmax, sketch, sketch_scale, proj, sel,
                                            sel_cnt, out, lse, append, w, st);
    if (e != cudaErrorNotSupported) return e;
  }
  if (use_sched(p, append)) {
    const cudaError_t e = spg::launch_sched(p, q, k_pool, v_pool, k_scale, v_scale, page_table,
                                            seq_lens, minmax, sketch, sketch_scale, proj, sel,
                                            sel_cnt, out, lse, append, w, st);
    if (e != cudaErrorNotSupported) return e;
  }
  if (append && p.selector != SPG_SEL_PROBE) {  // the probe selector keeps no metadata
    const cudaError_t e = spg::launch_meta_update(p, k_pool, k_scale, page_table, seq_lens, 0,
                                                  minmax, const_cast<uint8_t*>(sketch),
                                                  const_cast<float*>(sketch_scale), proj, w.err,
                                                  st);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = spg::launch_select(p, q, page_table, seq_lens, minmax, sketch, sketch_scale,
                                     proj, w.scores, sel, sel_cnt, w, st);
  if (e == cudaSuccess)
    e = spg::launch_attention(p, q, k_pool, v_pool, k_scale, v_scale, page_table, seq_lens, sel,
                              sel_cnt, out, lse, w, st);
  return e;
}

spg_status check_kv(const spg_params* p, const void* k_pool, const void* v_pool,
                    const void* k_scale, const void* v_scale) {
  if (!ok_ptr(k_pool) || !ok_ptr(v_pool)) return SPG_EINVAL;
  if (p->kv_dtype == SPG_I8 && (!ok_ptr(k_scale) || !ok_ptr(v_scale))) return SPG_EINVAL;
  return SPG_OK;
}

}  // namespace

extern "C" {

int32_t spg_abi_version(void) { return SPG_ABI_VERSION; }

const char* spg_status_str(int32_t s) {
  switch (s) {
    case SPG_OK: return "ok";
    case SPG_EINVAL: return "invalid argument";
    case SPG_EUNSUPPORTED: return "unsupported configuration";
    case SPG_ECUDA: return "CUDA launch error";
    case SPG_EWORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

// largest K + V (+ scales) bytes of one page of one kv-head
constexpr int64_t kMaxPageBytes = 34 * 1024;

spg_status spg_validate(const spg_params* p) {
  if (!p) return SPG_EINVAL;
  if (p->batch < 1 || p->num_q_heads < 1 || p->num_kv_heads < 1) return SPG_EINVAL;
  if (p->num_q_heads % p->num_kv_heads) return SPG_EINVAL;
  if (p->head_dim < 32 || p->head_dim % 32) return SPG_EINVAL;
  if (p->page_size < 8 || p->page_size > 128 || (p->page_size & (p->page_size - 1)))
    return SPG_EINVAL;
  if (p->num_phys_pages < 1 || p->max_pages_per_seq < 1) return SPG_EINVAL;
  if (static_cast<int64_t>(p->max_pages_per_seq) * p->page_size > INT32_MAX) return SPG_EINVAL;
  if (p->kv_dtype < SPG_F16 || p->kv_dtype > SPG_I8) return SPG_EINVAL;
  if (p->q_dtype != SPG_F16 && p->q_dtype != SPG_BF16) return SPG_EINVAL;
  if (p->kv_dtype != SPG_I8 && p->q_dtype != p->kv_dtype) return SPG_EINVAL;
  if (p->selector < SPG_SEL_QUEST || p->selector > SPG_SEL_PROBE) return SPG_EINVAL;
  if (p->n_probe < 0) return SPG_EINVAL;
  if (!(p->softmax_scale >= 0.f) || std::isinf(p->softmax_scale)) return SPG_EINVAL;
  if (!(p->top_p >= 0.f && p->top_p <= 1.f) || p->min_pages < 0) return SPG_EINVAL;
  if (p->selector != SPG_SEL_ALL) {
    if (p->n_sink_pages < 0 || p->n_recent_pages < 0) return SPG_EINVAL;
    if (p->token_budget < p->page_size || p->token_budget % p->page_size) return SPG_EINVAL;
    if (spg::n_sel_pages(*p) < p->n_sink_pages + p->n_recent_pages) return SPG_EINVAL;
  }
  if (p->selector == SPG_SEL_SKETCH_INT4) {
    if (p->sketch_dim != 16) return SPG_EINVAL;
    if (p->n_recent_pages < 1) return SPG_EINVAL;  // the open tail block is never scored
  }
  // valid, but not built
  const int G = p->num_q_heads / p->num_kv_heads;
  if (p->head_dim != 64 && p->head_dim != 128) return SPG_EUNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8) return SPG_EUNSUPPORTED;
  if (p->selector == SPG_SEL_PROBE && p->kv_dtype == SPG_I8) return SPG_EUNSUPPORTED;
  // the tensor-core consumers take 16-token tiles of a staged page, and a
  // ring of four stages must hold four pages (K, V and int8 scales)
  if (p->page_size < 16) return SPG_EUNSUPPORTED;
  {
    const int64_t elem = p->kv_dtype == SPG_I8 ? 1 : 2;
    const int64_t page_bytes = 2 * static_cast<int64_t>(p->page_size) * p->head_dim * elem +
                               (p->kv_dtype == SPG_I8 ? 4 * p->page_size : 0);
    if (page_bytes > kMaxPageBytes) return SPG_EUNSUPPORTED;
  }
  if (p->selector != SPG_SEL_ALL && p->max_pages_per_seq > spg::kMaxTopkPages)
    return SPG_EUNSUPPORTED;
  if (p->max_pages_per_seq > spg::kMaxSplits * 1024) return SPG_EUNSUPPORTED;
  // the adaptive budget runs where the selection's keys sit in shared memory
  if (p->selector != SPG_SEL_ALL && p->top_p > 0.f &&
      (spg::n_sel_pages(*p) > spg::kMaxTopPPages || p->max_pages_per_seq > 8192))
    return SPG_EUNSUPPORTED;
  return SPG_OK;
}

spg_status spg_workspace_size(const spg_params* p, size_t* bytes) {
  const spg_status s = spg_validate(p);
  if (s != SPG_OK) return s;
  if (!bytes) return SPG_EINVAL;
  *bytes = spg::workspace_bytes(*p);
  return SPG_OK;
}

spg_status sparse_page_meta_update(const spg_params* p, const void* k_pool, const void* k_scale,
                                   const int32_t* page_table, const int32_t* seq_lens,
                                   int32_t rebuild, void* minmax, uint8_t* sketch,
                                   float* sketch_scale, const float* proj, void* ws,
                                   size_t ws_bytes, spg_stream_t stream) {
  spg_status s = spg_validate(p);
  if (s != SPG_OK) return s;
  if (!ok_ptr(k_pool) || !ok_ptr(page_table) || !ok_ptr(seq_lens)) return SPG_EINVAL;
  if (p->kv_dtype == SPG_I8 && !ok_ptr(k_scale)) return SPG_EINVAL;
  if ((s = check_meta_inputs(p, minmax, sketch, sketch_scale, proj)) != SPG_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != SPG_OK) return s;
  const Workspace w = spg::carve_workspace(*p, ws);
  if (p->selector == SPG_SEL_PROBE) return SPG_OK;  // no metadata to keep
  return cuda_status(spg::launch_meta_update(*p, k_pool, k_scale, page_table, seq_lens, rebuild,
                                             minmax, sketch, sketch_scale, proj, w.err,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

spg_status sparse_page_score(const spg_params* p, const void* q, const int32_t* page_table,
                             const int32_t* seq_lens, const void* minmax, const uint8_t* sketch,
                             const float* sketch_scale, const float* proj, float* scores, void* ws,
                             size_t ws_bytes, spg_stream_t stream) {
  spg_status s = spg_validate(p);
  if (s != SPG_OK) return s;
  if (!ok_ptr(q) || !ok_ptr(page_table) || !ok_ptr(seq_lens) || !ok_ptr(scores)) return SPG_EINVAL;
  if ((s = check_meta_inputs(p, minmax, sketch, sketch_scale, proj)) != SPG_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != SPG_OK) return s;
  const Workspace w = spg::carve_workspace(*p, ws);
  return cuda_status(spg::launch_select(*p, q, page_table, seq_lens, minmax, sketch, sketch_scale,
                                        proj, scores, nullptr, nullptr, w,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

spg_status sparse_page_select(const spg_params* p, const void* q, const int32_t* page_table,
                              const int32_t* seq_lens, const void* minmax, const uint8_t* sketch,
                              const float* sketch_scale, const float* proj, int32_t* sel,
                              int32_t* sel_cnt, void* ws, size_t ws_bytes, spg_stream_t stream) {
  spg_status s = spg_validate(p);
  if (s != SPG_OK) return s;
  if (!ok_ptr(q) || !ok_ptr(page_table) || !ok_ptr(seq_lens) || !ok_ptr(sel) || !ok_ptr(sel_cnt))
    return SPG_EINVAL;
  if ((s = check_meta_inputs(p, minmax, sketch, sketch_scale, proj)) != SPG_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != SPG_OK) return s;
  const Workspace w = spg::carve_workspace(*p, ws);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(spg::launch_select(*p, q, page_table, seq_lens, minmax, sketch, sketch_scale,
                                        proj, w.scores, sel, sel_cnt, w, st));
}

spg_status sparse_decode_attention(const spg_params* p, const void* q, const void* k_pool,
                                   const void* v_pool, const void* k_scale, const void* v_scale,
                                   const int32_t* page_table, const int32_t* seq_lens,
                                   const int32_t* sel, const int32_t* sel_cnt, float* out,
                                   float* lse, void* ws, size_t ws_bytes, spg_stream_t stream) {
  spg_status s = spg_validate(p);
  if (s != SPG_OK) return s;
  if (p->selector == SPG_SEL_ALL) return SPG_EINVAL;  // needs a token budget for sel's shape
  if (!ok_ptr(q) || !ok_ptr(page_table) || !ok_ptr(seq_lens) || !ok_ptr(sel) ||
      !ok_ptr(sel_cnt) || !ok_ptr(out) || (lse && !aligned16(lse)))
    return SPG_EINVAL;
  if ((s = check_kv(p, k_pool, v_pool, k_scale, v_scale)) != SPG_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != SPG_OK) return s;
  const Workspace w = spg::carve_workspace(*p, ws);
  return cuda_status(spg::launch_attention(*p, q, k_pool, v_pool, k_scale, v_scale, page_table,
                                           seq_lens, sel, sel_cnt, out, lse, w,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

spg_status sparse_decode_select_attend(const spg_params* p, const void* q, const void* k_pool,
                                       const void* v_pool, const void* k_scale,
                                       const void* v_scale, const int32_t* page_table,
                                       const int32_t* seq_lens, const void* minmax,
                                       const uint8_t* sketch, const float* sketch_scale,
                                       const float* proj, int32_t* sel, int32_t* sel_cnt,
                                       float* out, float* lse, void* ws, size_t ws_bytes,
                                       spg_stream_t stream) {
  spg_status s = spg_validate(p);
  if (s != SPG_OK) return s;
  if (!ok_ptr(q) || !ok_ptr(page_table) || !ok_ptr(seq_lens) || !ok_ptr(sel) ||
      !ok_ptr(sel_cnt) || !ok_ptr(out) || (lse && !aligned16(lse)))
    return SPG_EINVAL;
  if ((s = check_meta_inputs(p, minmax, sketch, sketch_scale, proj)) != SPG_OK) return s;
  if ((s = check_kv(p, k_pool, v_pool, k_scale, v_scale)) != SPG_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != SPG_OK) return s;
  const Workspace w = spg::carve_workspace(*p, ws);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(select_attend(*p, q, k_pool, v_pool, k_scale, v_scale, page_table, seq_lens,
                                   const_cast<void*>(minmax), sketch, sketch_scale, proj, sel,
                                   sel_cnt, out, lse, 0, w, st));
}

spg_status sparse_decode_step(const spg_params* p, const void* q, const void* k_pool,
                              const void* v_pool, const void* k_scale, const void* v_scale,
                              const int32_t* page_table, const int32_t* seq_lens, void* minmax,
                              uint8_t* sketch, float* sketch_scale, const float* proj,
                              int32_t* sel, int32_t* sel_cnt, float* out, float* lse, void* ws,
                              size_t ws_bytes, spg_stream_t stream) {
  spg_status s = spg_validate(p);
  if (s != SPG_OK) return s;
  if (!ok_ptr(q) || !ok_ptr(page_table) || !ok_ptr(seq_lens) || !ok_ptr(sel) ||
      !ok_ptr(sel_cnt) || !ok_ptr(out) || (lse && !aligned16(lse)))
    return SPG_EINVAL;
  if ((s = check_meta_inputs(p, minmax, sketch, sketch_scale, proj)) != SPG_OK) return s;
  if ((s = check_kv(p, k_pool, v_pool, k_scale, v_scale)) != SPG_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != SPG_OK) return s;
  const Workspace w = spg::carve_workspace(*p, ws);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  int append_inside = (use_sched(*p, 1) || use_fused(*p, 1)) ? 1 : 0;
  if (!append_inside && p->selector != SPG_SEL_PROBE)
    e = spg::launch_meta_update(*p, k_pool, k_scale, page_table, seq_lens, 0, minmax, sketch,
                                sketch_scale, proj, w.err, st);
  if (e == cudaSuccess)
    e = select_attend(*p, q, k_pool, v_pool, k_scale, v_scale, page_table, seq_lens, minmax,
                      sketch, sketch_scale, proj, sel, sel_cnt, out, lse, append_inside, w, st);
  return cuda_status(e);
}

spg_status dense_decode_attention(const spg_params* p, const void* q, const void* k_pool,
                                  const void* v_pool, const void* k_scale, const void* v_scale,
                                  const int32_t* page_table, const int32_t* seq_lens, float* out,
                                  float* lse, void* ws, size_t ws_bytes, spg_stream_t stream) {
  spg_status s = spg_validate(p);
  if (s != SPG_OK) return s;
  if (!ok_ptr(q) || !ok_ptr(page_table) || !ok_ptr(seq_lens) || !ok_ptr(out) ||
      (lse && !aligned16(lse)))
    return SPG_EINVAL;
  if ((s = check_kv(p, k_pool, v_pool, k_scale, v_scale)) != SPG_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != SPG_OK) return s;
  const Workspace w = spg::carve_workspace(*p, ws);
  return cuda_status(spg::launch_attention(*p, q, k_pool, v_pool, k_scale, v_scale, page_table,
                                           seq_lens, nullptr, nullptr, out, lse, w,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

spg_status sparse_page_sketch_dots(const spg_params* p, const void* q, const int32_t* seq_lens,
                                   const uint8_t* sketch, const float* proj, int32_t* qc,
                                   float* sq, int32_t* dots, void* ws, size_t ws_bytes,
                                   spg_stream_t stream) {
  spg_status s = spg_validate(p);
  if (s != SPG_OK) return s;
  if (p->selector != SPG_SEL_SKETCH_INT4) return SPG_EINVAL;
  if (!ok_ptr(q) || !ok_ptr(seq_lens) || !ok_ptr(sketch) || !ok_ptr(proj) || !ok_ptr(qc) ||
      !ok_ptr(sq) || !ok_ptr(dots))
    return SPG_EINVAL;
  if ((s = check_ws(p, ws, ws_bytes)) != SPG_OK) return s;
  const Workspace w = spg::carve_workspace(*p, ws);
  return cuda_status(spg::launch_sketch_dots(*p, q, seq_lens, sketch, proj, qc, sq, dots, w.err,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int32_t spg_prefer_dense(const spg_params* p, int32_t max_seq_len, float ratio) {
  if (spg_validate(p) != SPG_OK || p->selector == SPG_SEL_ALL || max_seq_len < 0) return 0;
  if (!(ratio > 0.f)) ratio = SPG_DENSE_BYPASS_RATIO;
  const int64_t pages = (static_cast<int64_t>(max_seq_len) + p->page_size - 1) / p->page_size;
  return static_cast<double>(pages) <= static_cast<double>(ratio) * spg::n_sel_pages(*p) ? 1 : 0;
}

const char* spg_step_kernel(const spg_params* p) {
  if (spg_validate(p) != SPG_OK) return nullptr;
  if (p->selector == SPG_SEL_ALL) return "k_attn";
  if (use_fused(*p, 1)) return "k_fused";
  if (use_sched(*p, 1)) return "k_sched";
  if (p->selector == SPG_SEL_PROBE) return "k_probe_select+k_attn";
  return p->selector == SPG_SEL_QUEST ? "k_quest_select+k_attn" : "k_sketch_select+k_attn";
}

int32_t spg_step_launches(const spg_params* p) {
  if (spg_validate(p) != SPG_OK) return 0;
  if (p->selector == SPG_SEL_ALL) return 1;
  if (use_sched(*p, 1) || use_fused(*p, 1)) return 1;
  // append (none for the probe selector), scoring (+ a separate selection
  // kernel past 8192 pages), attention
  return (p->selector == SPG_SEL_PROBE ? 2 : 3) + (p->max_pages_per_seq > 8192 ? 1 : 0);
}

spg_status spg_set_step_kernel(int32_t kernel) {
  if (kernel < 0 || kernel > 2) return SPG_EINVAL;
  g_step_pref.store(kernel);
  return SPG_OK;
}

spg_status spg_read_device_error(const void* ws, int32_t* bits, spg_stream_t stream) {
  if (!ok_ptr(ws) || !bits) return SPG_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SPG_ECUDA;
  if (cudaMemcpy(bits, ws, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPG_ECUDA;
  return SPG_OK;
}

spg_status spg_test_withhold_first_stage(void* ws, spg_stream_t stream) {
  if (!ok_ptr(ws)) return SPG_EINVAL;
  static const int32_t one = 1;
  return cuda_status(cudaMemcpyAsync(static_cast<uint8_t*>(ws) + 128, &one, sizeof(one),
                                     cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream)));
}

spg_status spg_clear_device_error(void* ws, spg_stream_t stream) {
  if (!ok_ptr(ws)) return SPG_EINVAL;
  return cuda_status(
      cudaMemsetAsync(ws, 0, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
