// Host-side launchers shared between the kernel files and the C ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spg.h"

namespace spg {

// Workspace carved into its regions (all device pointers).
struct Workspace {
  int32_t* err;     // error word (header)
  int32_t* hook;    // test hook (header, byte 128): see spg_test_withhold_first_stage
  int32_t* counters;  // [B][Hkv] split arrivals of the attention kernel; zero between calls
  int32_t* sel_counters;  // [B][Hkv] scoring CTAs done, for the fused selection; zero between calls
  float* scores;    // [B][Hkv][MP]
  float* pm;        // [B][Hq][kMaxSplits] running max (log2 domain)
  float* pl;        // [B][Hq][kMaxSplits] running sum
  float* pacc;      // [B][Hq][kMaxSplits][d] unnormalised output
  // the persistent scheduled step (spg_sched.cu)
  int32_t* sched_ctr;    // [8] queue counters (in the header); zero between calls
  int32_t* sched_flags;  // [4][B*Hkv] per-unit flags; zero between calls
  int2* slices;          // [B*Hkv][n_sel] (physical page, valid tokens) of the selection
  int32_t* iq;           // [B*Hkv][8] sketch index queries
};

size_t workspace_bytes(const spg_params& p);

// Tensor map of a K or V pool (rows = num_phys_pages * num_kv_heads *
// page_size rows of head_dim elements) through which one page of one kv-head
// lands in shared memory as head_dim * elem_bytes / 128 tiles of [page_size
// rows][128 bytes] (64 fp16/bf16 channels or 128 int8 ones each, 128-byte
// swizzle).  *whole_page: the map is 3-D and one copy (coordinates {0, row,
// 0}) brings the whole page; else it is 2-D and each tile is one copy
// (coordinates {64-channel slice start, row}).  False when the pool cannot be
// described (dtype, alignment, size) or the encoder is unavailable.
bool make_kv_tmap(CUtensorMap* map, const void* pool, int kv_dtype, long long rows, int head_dim,
                  int page_size, bool* whole_page);
Workspace carve_workspace(const spg_params& p, void* ws);

int n_sel_pages(const spg_params& p);
int device_sm_count();
int max_splits(const spg_params& p);

cudaError_t launch_meta_update(const spg_params& p, const void* k_pool, const void* k_scale,
                               const int32_t* page_table, const int32_t* seq_lens, int rebuild,
                               void* minmax, uint8_t* sketch, float* sketch_scale,
                               const float* proj, int32_t* err, cudaStream_t stream);

// Scores every candidate page into `scores`; with sel != nullptr also
// selects each unit's pages (inside the scoring launch, or in a separate
// selection kernel for very long page tables).
cudaError_t launch_select(const spg_params& p, const void* q, const int32_t* page_table,
                          const int32_t* seq_lens, const void* minmax, const uint8_t* sketch,
                          const float* sketch_scale, const float* proj, float* scores,
                          int32_t* sel, int32_t* sel_cnt, const Workspace& ws,
                          cudaStream_t stream);

// sel == nullptr -> dense (every page of every sequence)
cudaError_t launch_attention(const spg_params& p, const void* q, const void* k_pool,
                             const void* v_pool, const void* k_scale, const void* v_scale,
                             const int32_t* page_table, const int32_t* seq_lens,
                             const int32_t* sel, const int32_t* sel_cnt, float* out, float* lse,
                             const Workspace& ws, cudaStream_t stream);

// The sketch selector's index query codes / scale and per-token integer
// dots of every candidate block (sparse_page_sketch_dots).
cudaError_t launch_sketch_dots(const spg_params& p, const void* q, const int32_t* seq_lens,
                               const uint8_t* sketch, const float* proj, int32_t* qc, float* sq,
                               int32_t* dots, int32_t* err, cudaStream_t stream);

// The whole step in one cluster launch (see spg_fused.cu).  fused_supported
// says whether these parameters can take that path; launch_fused returns
// cudaErrorNotSupported, before launching, when the page layout does not fit
// its shared-memory plan.
bool fused_supported(const spg_params& p, int append);
// The whole step as one persistent launch with task queues (see
// spg_sched.cu); launch_sched returns cudaErrorNotSupported, before
// launching, when the parameters do not fit its plan.
bool sched_supported(const spg_params& p, int append);
cudaError_t launch_sched(const spg_params& p, const void* q, const void* k_pool,
                         const void* v_pool, const void* k_scale, const void* v_scale,
                         const int32_t* page_table, const int32_t* seq_lens, void* minmax,
                         const uint8_t* sketch, const float* sketch_scale, const float* proj,
                         int32_t* sel, int32_t* sel_cnt, float* out, float* lse, int append,
                         const Workspace& ws, cudaStream_t stream);
cudaError_t launch_fused(const spg_params& p, const void* q, const void* k_pool,
                         const void* v_pool, const void* k_scale, const void* v_scale,
                         const int32_t* page_table, const int32_t* seq_lens, void* minmax,
                         const uint8_t* sketch, const float* sketch_scale, const float* proj,
                         int32_t* sel, int32_t* sel_cnt, float* out, float* lse, int append,
                         const Workspace& ws, cudaStream_t stream);

}  // namespace spg
