// The whole decode step as one persistent, dynamically scheduled launch:
// page scoring, exact top-k, sparse flash-decoding, the log-sum-exp merge
// and the metadata append of the new token.
//
// Sources: Quest 完全拆解 (核心机制: the per-page bound; 关键性估计算法: the
// insert-time min/max; 三段式 kernel: estimate -> top-k -> approximate
// attention); SALS长序列推理优化 (QSI: index query, int4 index key, block
// log-sum-exp, exact top-k; SFAA: attention over the selected int8 blocks;
// AICPU Tiling: the work of a step cut into tasks by a cost model ahead of
// the compute, and a row split over several cores merged by a reduction);
// SequenceO1 close reading §2.4 / §3.3 (select and attend fused, only int32
// page ids between them).
//
// Why one launch with queues.  The work of a step is three dependent phases
// per (batch, kv-head) unit: scan the unit's metadata, select its pages,
// attend to them.  When every unit moves through the phases in lockstep
// (one group of CTAs per unit), the memory system idles while every unit
// selects at the same moment.  Here the units are decoupled: CTAs take
// scan tasks and attend tasks from global queues, in unit order, and a few
// CTAs select; a unit is selected as soon as its own scan is complete, while
// other units are still being scanned, and attended as soon as its
// selection is published, while later units are still being selected.
//
// Roles (the first n_selectors CTAs to start are selectors, the rest
// workers; a selector becomes a worker when no unit is left to select):
//  * worker, warp 4 (producer): takes scan tasks (one stage of up to R
//    metadata rows of one unit: one cp.async.bulk, plus the unit's query
//    rows), then, when none is left, attend tasks (4 x SPW stages of up to
//    PPS selected pages of one unit: one TMA tile copy per page for K and for
//    V, bulk copies of int8 scales), and writes each stage's descriptor;
//  * worker, warps 0-3 (consumers): stage k belongs to warp k % 4.  A scan
//    stage is scored (Quest on tensor cores, sketch one block per lane) and
//    its order-preserving keys stored in the workspace; the unit's counter
//    of scored rows is then advanced.  An attend stage runs flash-decoding
//    over its pages; at the end of a task the four warps merge their states
//    and write one partial (m, l, acc) of the unit; the task that completes a
//    unit merges all of its partials into out / lse;
//  * selector (the whole CTA): for each unit in turn (a global counter),
//    waits until the unit's rows are all scored, loads the keys, runs the
//    exact top-k (block_topk), adds the forced pages, writes sel / sel_cnt
//    and the (physical page, valid tokens) list the attend tasks read, then
//    publishes the unit (release flag) and applies the metadata append of the
//    new token (its page is forced: nothing in the step reads it).  For the
//    sketch selector, the selectors first compute every scanned unit's index
//    query (one unit per warp) and publish it for the scan tasks.
// No CTA waits for a CTA that may not be running: a worker takes an attend
// task only when every scan task has been taken (by running CTAs, which
// finish them without waiting), so every unit's scan completes; selectors
// are running CTAs by construction.  Every wait is bounded (the error word
// gets SPG_DEVERR_TIMEOUT and the launch winds down).  The last CTA to
// leave resets the queue counters, and per-unit flags are reset by their
// last reader, so the workspace is ready for the next launch.
#include "spg_append.cuh"
#include "spg_attn_core.cuh"
#include "spg_internal.h"
#include "spg_select_core.cuh"

namespace spg {
namespace {

constexpr int kThreads = (kConsumerWarps + 2) * 32;  // 4 consumers, producer, auxiliary
constexpr int kMaxRows = 64;                         // metadata rows per scan stage
constexpr int kScanGroup = 8;                        // stages per scan task (one queue grab)
constexpr int kMaxPPS = 8;                           // pages per attend stage
constexpr int kStageTarget = 16 * 1024;              // bytes of a stage, about
constexpr int kSchedMaxBatch = 256;
constexpr int kSchedMaxPages = 8192;
constexpr uint64_t kSpinNs = 250ull * 1000 * 1000;  // longest wait for another CTA

// queue counters in the workspace (zero between launches)
enum { kScanNext = 0, kAttNext, kRoleNext, kSelNext, kIqNext, kExitCnt, kAbort, kNumCtr };
// per-unit flags, [4][units]
enum { kScanDone = 0, kReady, kAttDone, kIqReady };
// stage kinds
enum { kStScan = 1, kStAtt = 2, kStSkip = 3, kStEnd = 4 };

struct StageDesc {
  int kind, unit, first, count;  // scan: first logical page, rows; attend: first list index, pages
  int split, tpos;               // attend: task index in the unit, stage position in the task
  int qc[4];                     // sketch scan: the unit's int8 index query (packed for dp4a)
  float sq;                      //   and its scale
  int pad[3];
};

struct SchedArgs {
  CUtensorMap tmk, tmv;  // K / V pools as page tiles (tensor-core consumers)
  int whole_page;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const __half* k_scale;
  const __half* v_scale;
  const int32_t* page_table;
  const int32_t* seq_lens;
  void* minmax;
  uint8_t* sketch;
  float* sketch_scale;
  const float* proj;
  int32_t* sel;
  int32_t* sel_cnt;
  float* out;
  float* lse;
  int32_t* err;
  int32_t* ctr;     // [kNumCtr]
  int32_t* uflags;  // [4][units]
  uint32_t* keys;   // [units][MP]
  int2* slices;     // [units][n_sel] (physical page, valid tokens)
  int32_t* iq;      // [units][8]
  float* pm;
  float* pl;
  float* pacc;
  int B, Hkv, S, MP, n_phys, n_sink, n_recent, n_sel, append;
  int units, R, PPS, SPW, stages, n_selectors;
  uint32_t stage_bytes, row_bytes, page_bytes, qbytes;
  uint32_t off_qbuf, off_merge;                            // worker layout
  uint32_t off_spt, off_ssel, off_topk, off_sqbar, off_sP, off_tps;  // selector layout
  uint32_t off_fixed;                                       // both roles
  int pt_cached;
  float scale_log2, inv_sqrt_d;
  float top_p, tau;  // adaptive budget (top_p 0: off)
  int min_pages;
};

// fixed region (after the role-specific union)
struct FixedSmem {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t tbar;   // the 4 consumer warps at the end of an attend task
  uint64_t ptbar;  // selector: the page-table row has landed
  StageDesc desc[kMaxStages];
  int nv[kMaxStages][kMaxPPS];
  float rsc[kMaxStages][kMaxRows];
  int L[kSchedMaxBatch];
  int spref[kSchedMaxBatch + 1];  // scan tasks before batch b (all its heads)
  int apref[kSchedMaxBatch + 1];  // attend tasks before batch b
  float red[kThreads / 32];
  int role, unit, last, pad;
};

struct BInfo {
  int L, P, lo, hi, nc, k_top, cnt;
};

__device__ __forceinline__ BInfo binfo(int L, int S, int n_sink, int n_recent, int n_sel) {
  BInfo r;
  r.L = L;
  r.P = (L + S - 1) / S;
  r.lo = min(n_sink, r.P);
  r.hi = max(r.P - n_recent, r.lo);
  r.nc = r.hi - r.lo;
  const int nf = r.P - r.nc;
  r.k_top = min(max(n_sel - nf, 0), r.nc);
  r.cnt = r.lo + r.k_top + (r.P - r.hi);
  return r;
}
// a unit's candidates are scored when the top-k or the adaptive budget needs them
__device__ __forceinline__ bool needs_scan(const BInfo& i, bool adapt) {
  return i.k_top > 0 && (i.k_top < i.nc || adapt);
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int32_t* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void red_release_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_acq_rel_add(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool aborted(const SchedArgs& a) {
  return *reinterpret_cast<volatile int32_t*>(a.ctr + kAbort) != 0;
}
__device__ __forceinline__ void set_abort(const SchedArgs& a) {
  record_error(a.err, SPG_DEVERR_TIMEOUT);
  atomicExch(a.ctr + kAbort, 1);
}

// Waits until *p >= target (acquire).  Bounded: gives up after kSpinNs, or
// at once when another wait of this launch has given up; false then.
__device__ bool spin_geq(const SchedArgs& a, const int32_t* p, int target) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = globaltimer();
  uint32_t ns = 32;
  for (;;) {
    __nanosleep(ns);
    if (ld_acquire(p) >= target) return true;
    if (ns < 256) ns <<= 1;
    if (aborted(a)) return false;
    if (globaltimer() - t0 > kSpinNs) {
      set_abort(a);
      return false;
    }
  }
}

// largest b with pref[b] <= t (pref non-decreasing, pref[0] = 0 <= t)
__device__ __forceinline__ int find_batch(const int* pref, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// the 4 consumer warps at one point of an attend task (mbarrier of count 4,
// bounded wait); false when the wait ran out
__device__ __forceinline__ bool task_sync(FixedSmem& f, uint32_t& phase, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(&f.tbar);
  const bool ok = mbar_wait_bounded(&f.tbar, phase);
  phase ^= 1u;
  return ok;
}

template <typename T, typename TQ, int D, int G, int SEL>
__global__ void __launch_bounds__(kThreads) k_sched(const __grid_constant__ SchedArgs a) {
  constexpr int CW = kConsumerWarps;
  constexpr int CONS = !is_i8<T>() ? 1 : ((D == 128 && std::is_same<TQ, __half>::value) ? 2 : 0);
  constexpr bool MMA = CONS != 0;
  using TM = std::conditional_t<is_i8<T>(), TQ, T>;  // Quest metadata type
  using Consumer = std::conditional_t<
      CONS == 1, AttnMma<T, D, G>,
      std::conditional_t<CONS == 2, AttnMmaI8<G>, AttnConsumer<T, D, G, 1>>>;

  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  FixedSmem& f = *reinterpret_cast<FixedSmem*>(smem + a.off_fixed);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.B, Hkv = a.Hkv, S = a.S, MP = a.MP, Hq = Hkv * G;
  const int STAGES = a.stages, R = a.R, PPS = a.PPS, SPW = a.SPW, PPT = 4 * a.SPW * a.PPS;
  int32_t* scan_done = a.uflags + kScanDone * a.units;
  int32_t* ready = a.uflags + kReady * a.units;
  int32_t* att_done = a.uflags + kAttDone * a.units;
  int32_t* iq_ready = a.uflags + kIqReady * a.units;

  if (tid == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&f.full[s], 1);
      mbar_init(&f.empty[s], 1);
    }
    mbar_init(&f.tbar, CW);
    mbar_init(&f.ptbar, 1);
    mbar_fence_init();
  }
  if constexpr (MMA) {
    if (tid == CW * 32) {
      tma_prefetch_desc(&a.tmk);
      tma_prefetch_desc(&a.tmv);
    }
  }
  pdl_wait();

  // per-batch task counts and their prefix sums (warp 0)
  if (warp == 0) {
    int cs = 0, ca = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int ns = 0, na = 0;
      if (b < B) {
        int L = a.seq_lens[b];
        if (L < 0 || L > MP * S) {
          record_error(a.err, SPG_DEVERR_SEQ_LEN);
          L = 0;
        }
        f.L[b] = L;
        const BInfo bi = binfo(L, S, a.n_sink, a.n_recent, a.n_sel);
        ns = needs_scan(bi, a.top_p > 0.f) ? (bi.nc + kScanGroup * R - 1) / (kScanGroup * R) * Hkv : 0;
        na = (bi.cnt + PPT - 1) / PPT * Hkv;
      }
      int is = ns, ia = na;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int xs = __shfl_up_sync(0xffffffffu, is, o), xa = __shfl_up_sync(0xffffffffu, ia, o);
        if (lane >= o) {
          is += xs;
          ia += xa;
        }
      }
      if (b < B) {
        f.spref[b + 1] = cs + is;
        f.apref[b + 1] = ca + ia;
      }
      cs += __shfl_sync(0xffffffffu, is, 31);
      ca += __shfl_sync(0xffffffffu, ia, 31);
    }
    if (lane == 0) {
      f.spref[0] = 0;
      f.apref[0] = 0;
      f.role = atomicAdd(a.ctr + kRoleNext, 1) < a.n_selectors ? 1 : 0;
    }
  }
  __syncthreads();
  const int n_scan_tasks = f.spref[B], n_att_tasks = f.apref[B];

  // ================================================================ selector
  if (f.role) {
    const int nt = blockDim.x;
    if constexpr (SEL == 1) {
      // index queries of the units that are scanned: the group-mean query,
      // projected and quantised to int8 (QSI step 1), one unit per warp,
      // every product rounded and the sum taken in channel order
      float* s_P = reinterpret_cast<float*>(smem + a.off_sP);
      float* s_qbar = reinterpret_cast<float*>(smem + a.off_sqbar) + warp * D;
      for (int i = tid; i < D * 16 / 4; i += nt)
        reinterpret_cast<float4*>(s_P)[i] = __ldg(reinterpret_cast<const float4*>(a.proj) + i);
      __syncthreads();
      for (;;) {
        int u = 0;
        if (lane == 0) u = atomicAdd(a.ctr + kIqNext, 1);
        u = __shfl_sync(0xffffffffu, u, 0);
        if (u >= a.units) break;
        const int b = u / Hkv, h = u % Hkv;
        if (!needs_scan(binfo(f.L[b], S, a.n_sink, a.n_recent, a.n_sel), a.top_p > 0.f)) continue;
        const TQ* qb = static_cast<const TQ*>(a.q) + (static_cast<size_t>(b) * Hq + h * G) * D;
        int c[4];
        float sq;
        sketch_index_query_warp<TQ>(qb, G, D, s_P, s_qbar, lane, c, sq);
        if (lane == 0) {
          int32_t* dst = a.iq + static_cast<size_t>(u) * 8;
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[k] = c[k];
          dst[4] = __float_as_int(sq);
          __threadfence();
          st_release(iq_ready + u, 1);
        }
      }
      __syncthreads();
    }

    uint32_t* s_keys = reinterpret_cast<uint32_t*>(smem);
    int* s_pt = reinterpret_cast<int*>(smem + a.off_spt);
    int* s_sel = reinterpret_cast<int*>(smem + a.off_ssel);
    TopkShared& tk = *reinterpret_cast<TopkShared*>(smem + a.off_topk);
    uint32_t ptphase = 0;
    for (;;) {
      if (tid == 0) f.unit = atomicAdd(a.ctr + kSelNext, 1);
      __syncthreads();
      const int u = f.unit;
      __syncthreads();
      if (u >= a.units) break;
      const int b = u / Hkv, h = u % Hkv;
      const BInfo bi = binfo(f.L[b], S, a.n_sink, a.n_recent, a.n_sel);
      const int lo = bi.lo, hi = bi.hi, nc = bi.nc, P = bi.P;
      int k_top = bi.k_top;
      const bool scan = needs_scan(bi, a.top_p > 0.f);
      const bool pt_smem = a.pt_cached && P > 0;
      if (pt_smem && tid == 0) {
        // the unit's page-table row, while the scan runs
        const uint32_t bytes = (static_cast<uint32_t>(P) * 4u + 15u) & ~15u;
        mbar_expect_tx(&f.ptbar, bytes);
        bulk_g2s(s_pt, a.page_table + static_cast<size_t>(b) * MP, bytes, &f.ptbar);
        mbar_arrive(&f.ptbar);
      }
      for (int i = tid; i < 512; i += nt) reinterpret_cast<int4*>(tk.hist)[i] = make_int4(0, 0, 0, 0);
      if (scan) {
        if (tid == 0) spin_geq(a, scan_done + u, nc);
        __syncthreads();
        (void)ld_acquire(scan_done + u);
        // the keys into shared memory, eight loads per thread in flight, and
        // their min / max on the way
        const uint32_t* kg = a.keys + static_cast<size_t>(u) * MP + lo;
        uint32_t kmn = 0xffffffffu, kmx = 0u;
        for (int i0 = 0; i0 < nc; i0 += 8 * nt) {
          uint32_t v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = i0 + j * nt + tid;
            v[j] = i < nc ? __ldcg(kg + i) : 0u;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = i0 + j * nt + tid;
            if (i < nc) {
              s_keys[i] = v[j];
              kmn = min(kmn, v[j]);
              kmx = max(kmx, v[j]);
            }
          }
        }
        kmn = __reduce_min_sync(0xffffffffu, kmn);
        kmx = __reduce_max_sync(0xffffffffu, kmx);
        if (lane == 0) {
          f.red[warp] = __uint_as_float(kmn);
          reinterpret_cast<uint32_t*>(tk.wb)[warp] = kmx;
        }
        __syncthreads();
        if (tid == 0) {
          uint32_t mn = 0xffffffffu, mx = 0u;
          for (int w2 = 0; w2 < nt / 32; ++w2) {
            mn = min(mn, __float_as_uint(f.red[w2]));
            mx = max(mx, reinterpret_cast<const uint32_t*>(tk.wb)[w2]);
          }
          tk.kmin = mn;
          tk.kmax = mx;
        }
        __syncthreads();
        if (k_top < nc)
          block_topk(s_keys, nc, k_top, lo, s_sel + lo, tk, true, true);
      }
      for (int i = tid; i < lo; i += nt) s_sel[i] = i;
      if (k_top == nc)
        for (int i = tid; i < nc; i += nt) s_sel[lo + i] = lo + i;
      if (scan && a.top_p > 0.f) {  // the adaptive budget trims the chosen candidates
        __syncthreads();
        uint32_t* tps = reinterpret_cast<uint32_t*>(smem + a.off_tps);
        k_top = topp_trim(s_keys, nc, s_sel + lo, k_top, lo, a.tau, a.top_p, a.min_pages, tps,
                          reinterpret_cast<int*>(tps + kTopPScratchWords),
                          reinterpret_cast<float*>(tps + kTopPScratchWords + 40));
      }
      __syncthreads();
      for (int j = tid; j < P - hi; j += nt) s_sel[lo + k_top + j] = hi + j;
      const int count = lo + k_top + (P - hi);
      __syncthreads();
      if (pt_smem) {
        if (!mbar_wait_bounded(&f.ptbar, ptphase) && tid == 0) set_abort(a);
        ptphase ^= 1u;
      }
      // the selection, and the list the attend tasks read
      int32_t* gsel = a.sel + static_cast<size_t>(u) * a.n_sel;
      int2* gsl = a.slices + static_cast<size_t>(u) * a.n_sel;
      for (int i = tid; i < a.n_sel; i += nt) {
        const int lp = i < count ? s_sel[i] : -1;
        gsel[i] = lp;
        if (i < count) {
          int ph = -1, nv = 0;
          if (lp < 0 || lp >= P) {
            record_error(a.err, SPG_DEVERR_SEL);
          } else {
            ph = pt_smem ? s_pt[lp] : a.page_table[static_cast<size_t>(b) * MP + lp];
            if (ph < 0 || ph >= a.n_phys) {
              record_error(a.err, SPG_DEVERR_PAGE_ID);
              ph = -1;
            } else {
              nv = min(S, bi.L - lp * S);
            }
          }
          gsl[i] = make_int2(ph, nv);
        }
      }
      if (count == 0) {  // an empty sequence: out = 0, lse = -inf
        for (int idx = tid; idx < G * D; idx += nt) {
          const size_t row = static_cast<size_t>(b) * Hq + h * G + idx / D;
          a.out[row * D + idx % D] = 0.f;
          if (idx % D == 0 && a.lse) a.lse[row] = -INFINITY;
        }
      }
      if (tid == 0) a.sel_cnt[u] = count;
      // the CTA barrier orders every thread's stores before thread 0's
      // release store, which publishes them all to the GPU
      __syncthreads();
      if (tid == 0) {
        if (scan) {
          scan_done[u] = 0;
          if constexpr (SEL == 1) iq_ready[u] = 0;
        }
        if (count > 0) st_release(ready + u, 1);
      }
      // the metadata append of the token at L - 1: its page is forced, so
      // no scan or attend task of this step reads what is written
      if (a.append && bi.L > 0) {
        if constexpr (SEL == 0) {
          if (warp == 0) {
            if constexpr (is_i8<T>())
              minmax_append_warp_i8<TM, D>(static_cast<const int8_t*>(a.k_pool), a.k_scale,
                                           a.page_table, static_cast<TM*>(a.minmax), a.err, Hkv, S,
                                           MP, a.n_phys, b, h, bi.L, lane);
            else
              minmax_append_warp<T, D>(static_cast<const T*>(a.k_pool), a.page_table,
                                       static_cast<T*>(a.minmax), a.err, Hkv, S, MP, a.n_phys, b,
                                       h, bi.L, lane);
          }
        } else {
          if (bi.L % S == 0)
            sketch_block_cta<T, D>(static_cast<const T*>(a.k_pool), a.k_scale, a.page_table, a.proj,
                                   a.sketch, a.sketch_scale, a.err, Hkv, S, MP, a.n_phys, b, h,
                                   bi.L / S - 1, f.red);
        }
      }
      __syncthreads();
    }
    // the ring now takes asynchronous copies where generic stores were
    fence_proxy_async();
    __syncthreads();
  }

  // ================================================================== worker
  uint8_t* ring = smem;
  uint8_t* qbuf = smem + a.off_qbuf;
  const uint32_t sbytes = a.stage_bytes, rb = a.row_bytes, pbytes = a.page_bytes;
  if (warp == CW) {
    // ---------------------------------------------------------- producer
    int k = 0;
    bool ok = true;
    auto take_slot = [&](int kk) -> bool {
      bool w = true;
      if (lane == 0 && kk >= STAGES) w = mbar_wait_bounded(&f.empty[kk % STAGES], ((kk / STAGES) - 1) & 1);
      w = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      if (!w && lane == 0) set_abort(a);
      return w;
    };
    auto post_empty = [&](int kind) {
      if (ok) ok = take_slot(k);
      if (lane == 0) {
        StageDesc& d = f.desc[k % STAGES];
        d.kind = kind;
        d.count = 0;
        mbar_arrive(&f.full[k % STAGES]);
      }
      __syncwarp();
      ++k;
    };
    // scan tasks: up to kScanGroup stages of R rows of one unit each, one
    // queue grab per task, the next grab in flight while a task is issued
    int t_next = 0;
    if (lane == 0) t_next = atomicAdd(a.ctr + kScanNext, 1);
    for (;;) {
      const int t = __shfl_sync(0xffffffffu, t_next, 0);
      if (t >= n_scan_tasks || !ok || aborted(a)) break;
      if (lane == 0) t_next = atomicAdd(a.ctr + kScanNext, 1);
      const int b = find_batch(f.spref, B, t);
      const BInfo bi = binfo(f.L[b], S, a.n_sink, a.n_recent, a.n_sel);
      const int per_head = (bi.nc + kScanGroup * R - 1) / (kScanGroup * R);
      const int loc = t - f.spref[b], h = loc / per_head, c = loc % per_head;
      const int u = b * Hkv + h;
      int qc_l = 0;  // sketch: this lane's word of the unit's index query (lanes 0-4)
      if constexpr (SEL == 1) {
        bool iqok = true;
        if (lane == 0) iqok = spin_geq(a, iq_ready + u, 1);
        iqok = __shfl_sync(0xffffffffu, iqok ? 1 : 0, 0) != 0;
        if (iqok) (void)ld_acquire(iq_ready + u);
        if (lane < 5 && iqok) qc_l = __ldcg(a.iq + static_cast<size_t>(u) * 8 + lane);
      }
      for (int g = 0; g < kScanGroup; ++g) {
        const int row0 = bi.lo + (c * kScanGroup + g) * R;
        if (row0 >= bi.hi) break;
        const int nr = min(R, bi.hi - row0);
        const int slot = k % STAGES;
        ok = take_slot(k);
        if (!ok) break;
        StageDesc& d = f.desc[slot];
        if constexpr (SEL == 1) {
          if (lane < 4) d.qc[lane] = qc_l;
          if (lane == 4) d.sq = __int_as_float(qc_l);
          const size_t lrow0 = static_cast<size_t>(u) * MP + row0;
          for (int r = lane; r < nr; r += 32) f.rsc[slot][r] = __ldg(a.sketch_scale + lrow0 + r);
        }
        if (lane == 0) {
          d.kind = kStScan;
          d.unit = u;
          d.first = row0;
          d.count = nr;
          const size_t lrow0 = static_cast<size_t>(u) * MP + row0;
          const uint8_t* src = SEL == 0 ? static_cast<const uint8_t*>(a.minmax) + lrow0 * rb
                                        : a.sketch + lrow0 * rb;
          uint32_t tx = static_cast<uint32_t>(nr) * rb;
          if constexpr (SEL == 0) tx += a.qbytes;
          mbar_expect_tx(&f.full[slot], tx);
          bulk_g2s(ring + static_cast<size_t>(slot) * sbytes, src, static_cast<uint32_t>(nr) * rb,
                   &f.full[slot]);
          if constexpr (SEL == 0)
            bulk_g2s(qbuf + static_cast<size_t>(slot) * a.qbytes,
                     static_cast<const TQ*>(a.q) + (static_cast<size_t>(b) * Hq + h * G) * D, a.qbytes,
                     &f.full[slot]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&f.full[slot]);
        ++k;
      }
    }
    // attend tasks start at a multiple of 4 stages (one stage per consumer
    // warp and task position)
    while (k % CW) post_empty(kStSkip);
    {
      const uint32_t tile = static_cast<uint32_t>(S) * D * sizeof(T);
      const uint32_t scb = is_i8<T>() ? static_cast<uint32_t>(S) * 2 : 0u;
      const uint64_t pol = policy_evict_first();
      int a_next = 0;
      if (lane == 0) a_next = atomicAdd(a.ctr + kAttNext, 1);
      for (;;) {
        const int t = __shfl_sync(0xffffffffu, a_next, 0);
        if (t >= n_att_tasks || !ok || aborted(a)) break;
        if (lane == 0) a_next = atomicAdd(a.ctr + kAttNext, 1);
        const int b = find_batch(f.apref, B, t);
        const BInfo bi = binfo(f.L[b], S, a.n_sink, a.n_recent, a.n_sel);
        const int per_head = (bi.cnt + PPT - 1) / PPT;
        const int loc = t - f.apref[b], h = loc / per_head, split = loc % per_head;
        const int u = b * Hkv + h;
        const int p0 = split * PPT;
        int p1 = min(p0 + PPT, bi.cnt);
        bool rdy = true;
        if (lane == 0) rdy = spin_geq(a, ready + u, 1);
        rdy = __shfl_sync(0xffffffffu, rdy ? 1 : 0, 0) != 0;
        if (rdy) {
          (void)ld_acquire(ready + u);
          // the adaptive budget may have kept fewer pages than the fixed one
          if (a.top_p > 0.f) p1 = min(p1, __ldcg(a.sel_cnt + u));
        }
        const int2* sl = a.slices + static_cast<size_t>(u) * a.n_sel;
        for (int j = 0; j < CW * SPW; ++j) {
          const int slot = k % STAGES;
          ok = ok && take_slot(k);
          const int pg0 = p0 + j * PPS;
          const int np = (ok && rdy) ? max(0, min(PPS, p1 - pg0)) : 0;
          uint8_t* stg = ring + static_cast<size_t>(slot) * sbytes;
          if (lane < np) {
            const int2 e = __ldcg(sl + pg0 + lane);
            const int ph = e.x;
            f.nv[slot][lane] = ph >= 0 ? e.y : 0;
            if (ph >= 0) {
              uint8_t* dst = stg + static_cast<size_t>(lane) * pbytes;
              const size_t row = static_cast<size_t>(ph) * Hkv + h;
              mbar_expect_tx(&f.full[slot], 2 * tile + 2 * scb);
              if constexpr (MMA) {
                const int y = static_cast<int>(row) * S;
                if (a.whole_page) {
                  tma_load_3d(dst, &a.tmk, 0, y, 0, &f.full[slot], pol);
                  tma_load_3d(dst + tile, &a.tmv, 0, y, 0, &f.full[slot], pol);
                } else {
                  constexpr int NT = D * static_cast<int>(sizeof(T)) / 128, EPT = 128 / sizeof(T);
#pragma unroll
                  for (int hf = 0; hf < NT; ++hf) {
                    tma_load_2d(dst + hf * S * 128, &a.tmk, hf * EPT, y, &f.full[slot], pol);
                    tma_load_2d(dst + tile + hf * S * 128, &a.tmv, hf * EPT, y, &f.full[slot], pol);
                  }
                }
              } else {
                bulk_g2s_hint(dst, static_cast<const T*>(a.k_pool) + row * S * D, tile, &f.full[slot], pol);
                bulk_g2s_hint(dst + tile, static_cast<const T*>(a.v_pool) + row * S * D, tile, &f.full[slot], pol);
              }
              if constexpr (is_i8<T>()) {
                bulk_g2s(dst + 2 * tile, a.k_scale + row * S, scb, &f.full[slot]);
                bulk_g2s(dst + 2 * tile + scb, a.v_scale + row * S, scb, &f.full[slot]);
              }
            }
          }
          if (lane == 0) {
            StageDesc& d = f.desc[slot];
            d.kind = kStAtt;
            d.unit = u;
            d.first = pg0;
            d.count = np;
            d.split = split;
            d.tpos = j;
            if (j < CW) {  // each warp's first stage of the task carries the query rows
              mbar_expect_tx(&f.full[slot], a.qbytes);
              bulk_g2s(qbuf + static_cast<size_t>(slot) * a.qbytes,
                       static_cast<const TQ*>(a.q) + (static_cast<size_t>(b) * Hq + h * G) * D,
                       a.qbytes, &f.full[slot]);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&f.full[slot]);
          ++k;
        }
      }
    }
    for (int e = 0; e < CW; ++e) post_empty(kStEnd);
  } else if (warp < CW) {
    // --------------------------------------------------------- consumers
    float* s_m = reinterpret_cast<float*>(smem + a.off_merge);  // [CW][G]
    float* s_l = s_m + CW * G;                                   // [CW][G]
    float* s_acc = s_l + CW * G;                                 // [CW][G][D]
    uint32_t tphase = 0;
    Consumer cons;
    for (int k = warp;; k += CW) {
      const int slot = k % STAGES;
      if (!mbar_wait_bounded(&f.full[slot], (k / STAGES) & 1)) {
        if (lane == 0) set_abort(a);
        break;
      }
      const StageDesc d = f.desc[slot];
      if (d.kind == kStEnd) break;
      const uint8_t* stg = ring + static_cast<size_t>(slot) * sbytes;
      if (d.kind == kStScan) {
        const int u = d.unit, nr = d.count;
        uint32_t* kout = a.keys + static_cast<size_t>(u) * MP;
        if constexpr (SEL == 0) {
          QuestMma<TM, D, G> qm;
          qm.init(reinterpret_cast<const TM*>(qbuf + static_cast<size_t>(slot) * a.qbytes), lane);
          const TM* st = reinterpret_cast<const TM*>(stg);
          for (int ti = 0; ti * 16 < nr; ++ti) {
            const int pt0 = d.first + ti * 16;
            float s0, s1;
            qm.tile(st + ti * 16 * 2 * D, pt0, lane, s0, s1);
            if ((lane & 3) == 0) {
              const int g = lane >> 2;
              if (ti * 16 + g < nr) kout[pt0 + g] = score_key(s0);
              if (ti * 16 + g + 8 < nr) kout[pt0 + g + 8] = score_key(s1);
            }
          }
        } else {
          const int qc[4] = {d.qc[0], d.qc[1], d.qc[2], d.qc[3]};
          const int qbias = sketch_query_bias(qc);
          if (lane < nr) {
            const float cz = __fmul_rn(__fmul_rn(d.sq, f.rsc[slot][lane]), a.inv_sqrt_d);
            const float sc = sketch_block_score_lane_t<0>(stg + lane * rb, S, qc, qbias, cz);
            kout[d.first + lane] = score_key(sc);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&f.empty[slot]);
        __syncwarp();  // the warp's keys, then the release add that publishes them
        if (lane == 0) red_release_add(scan_done + u, nr);
        continue;
      }
      if (d.kind == kStSkip) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&f.empty[slot]);
        continue;
      }
      // attend stage
      const int u = d.unit;
      if (d.tpos < CW)
        cons.init(reinterpret_cast<const TQ*>(qbuf + static_cast<size_t>(slot) * a.qbytes), a.scale_log2,
                  warp, lane);
      for (int i = 0; i < d.count; ++i) {
        const int nv = f.nv[slot][i];
        uint8_t* pg = ring + static_cast<size_t>(slot) * sbytes + static_cast<size_t>(i) * pbytes;
        if (nv > 0) {
          if constexpr (MMA)
            cons.consume(pg, S, nv, lane);
          else
            cons.consume(pg, S, nv);
        }
      }
      fence_proxy_async();  // reads (and zeroed slots) before the next copy into the slot
      __syncwarp();
      if (lane == 0) mbar_arrive(&f.empty[slot]);
      if (d.tpos / CW != SPW - 1) continue;
      // end of the task: the four warps' states -> one partial of the unit
      cons.fold();
      cons.store(s_m, s_l, s_acc, lane);
      bool sok = task_sync(f, tphase, lane);
      const int b = u / Hkv, h = u % Hkv;
      const int ct = warp * 32 + lane;  // 0 .. 127
      for (int idx = ct; idx < G * D; idx += CW * 32) {
        const int g = idx / D, c = idx % D;
        float M, Ls, A;
        lse_merge(s_m, s_l, s_acc, CW, G, D, g, c, M, Ls, A);
        const size_t prow = (static_cast<size_t>(b) * Hq + h * G + g) * kMaxSplits + d.split;
        __stcg(a.pacc + prow * D + c, A);
        if (c == 0) {
          __stcg(a.pm + prow, M);
          __stcg(a.pl + prow, Ls);
        }
      }
      sok = task_sync(f, tphase, lane) && sok;  // the partial, then the acq_rel count
      if (ct == 0) {
        const BInfo bi = binfo(f.L[b], S, a.n_sink, a.n_recent, a.n_sel);
        const int n_tasks = (bi.cnt + PPT - 1) / PPT;
        f.last = atom_acq_rel_add(att_done + u, 1) + 1 == n_tasks ? n_tasks : 0;
      }
      sok = task_sync(f, tphase, lane) && sok;
      const int n_last = f.last;
      if (n_last > 0) {
        // every partial of the unit is written: merge them (AICPU Tiling,
        // challenge 2: the reduction over the cores that shared a row)
        for (int idx = ct; idx < G * D; idx += CW * 32) {
          const int g = idx / D, c = idx % D;
          const size_t row = static_cast<size_t>(b) * Hq + h * G + g;
          const float* pm = a.pm + row * kMaxSplits;
          const float* pl = a.pl + row * kMaxSplits;
          const float* pa = a.pacc + row * kMaxSplits * D + c;
          // a running rescaled merge, eight partials' loads in flight at once
          float M = -INFINITY, A = 0.f, Ls = 0.f;
          for (int i0 = 0; i0 < n_last; i0 += 8) {
            float mv[8], lv[8], av[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const bool in = i0 + j < n_last;
              mv[j] = in ? __ldcg(pm + i0 + j) : -INFINITY;
              lv[j] = in ? __ldcg(pl + i0 + j) : 0.f;
              av[j] = in ? __ldcg(pa + static_cast<size_t>(i0 + j) * D) : 0.f;
            }
            float Mn = M;
#pragma unroll
            for (int j = 0; j < 8; ++j) Mn = fmaxf(Mn, mv[j]);
            if (Mn == -INFINITY) continue;
            const float r = exp2f(M - Mn);  // 0 while M is -inf
            A *= r;
            Ls *= r;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float w = exp2f(mv[j] - Mn);
              A = fmaf(av[j], w, A);
              Ls = fmaf(lv[j], w, Ls);
            }
            M = Mn;
          }
          a.out[row * D + c] = Ls > 0.f ? A / Ls : 0.f;
          if (c == 0 && a.lse) a.lse[row] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
        }
        if (ct == 0) {
          att_done[u] = 0;
          ready[u] = 0;
        }
      }
      sok = task_sync(f, tphase, lane) && sok;  // the merge area is free again
      if (!sok) {
        if (lane == 0) set_abort(a);
        break;
      }
    }
  }
  // the auxiliary warp has no worker role

  __syncthreads();
  pdl_trigger();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.ctr + kExitCnt, 1) == static_cast<int>(gridDim.x) - 1) {
      // the last CTA out: every queue is drained; ready for the next launch
      for (int i = 0; i < kNumCtr; ++i) a.ctr[i] = 0;
      __threadfence();
    }
  }
}

// ------------------------------------------------------------------ host side
template <typename T, typename TQ, int D, int G, int SEL>
cudaError_t sched_typed(const spg_params& p, SchedArgs a, cudaStream_t st) {
  constexpr bool MMA = !is_i8<T>() || (D == 128 && std::is_same<TQ, __half>::value);
  const int S = p.page_size;
  const int n_sel = n_sel_pages(p);
  // a page's K tile starts 1024-byte aligned for the swizzled TMA tiles
  const uint32_t pb = MMA ? (kv_stage_bytes<T, D>(S) + 1023u) & ~1023u : kv_stage_bytes<T, D>(S);
  using TM = std::conditional_t<is_i8<T>(), TQ, T>;  // Quest metadata type
  const uint32_t rb = SEL == 0 ? 2u * D * sizeof(TM) : static_cast<uint32_t>(S) * 8u;
  // Two ring slots per consumer warp (8 stages) of about kStageTarget / 2
  // bytes when a page fits in that, else one slot per warp of up to
  // kStageTarget: a warp then has its next stage in flight while it
  // consumes one.
  const bool deep = pb <= static_cast<uint32_t>(kStageTarget / 2);
  const int stages = deep ? 2 * kConsumerWarps : kConsumerWarps;
  const uint32_t target = deep ? kStageTarget / 2 : kStageTarget;
  int pps = 1;
  while (pps * 2 <= kMaxPPS && (pps * 2) * pb <= target) pps *= 2;
  int R;
  if (SEL == 0) {
    R = static_cast<int>(std::max<uint32_t>(pps * pb, target) / rb);
    R = (std::min(R, kMaxRows) / 16) * 16;  // whole 16-page tensor-core tiles
  } else {
    R = std::min<int>(32, std::max<uint32_t>(pps * pb, target) / rb);  // one block per lane
  }
  if (R < 1) return cudaErrorNotSupported;
  uint32_t sb = std::max<uint32_t>(pps * pb, static_cast<uint32_t>(R) * rb);
  sb = (sb + 1023u) & ~1023u;
  const uint32_t qbytes = static_cast<uint32_t>(G * D * sizeof(TQ));
  // worker layout
  const size_t off_qbuf = static_cast<size_t>(stages) * sb;
  const size_t off_merge = (off_qbuf + static_cast<size_t>(stages) * qbytes + 127) & ~size_t(127);
  const size_t worker_end = off_merge + sizeof(float) * kConsumerWarps * G * (D + 2);
  // selector layout
  const size_t mp = static_cast<size_t>(p.max_pages_per_seq);
  const size_t off_spt = (sizeof(uint32_t) * mp + 127) & ~size_t(127);
  const size_t off_ssel = (off_spt + sizeof(int) * mp + 127) & ~size_t(127);
  const size_t off_topk = (off_ssel + sizeof(int) * n_sel + 127) & ~size_t(127);
  const size_t off_sP = 0;  // index-query phase, before the keys are loaded
  const size_t off_sqbar = (sizeof(float) * D * 16 + 127) & ~size_t(127);
  const size_t off_tps = (off_topk + sizeof(TopkShared) + 127) & ~size_t(127);
  const size_t sel_end = std::max(off_tps + (p.top_p > 0.f ? sizeof(uint32_t) * (kTopPScratchWords + 80) : 0),
                                  off_sqbar + sizeof(float) * D * (kThreads / 32));
  const size_t off_fixed = (std::max(worker_end, sel_end) + 127) & ~size_t(127);
  const size_t smem = 1024 + off_fixed + sizeof(FixedSmem);
  if (smem > 227u * 1024u) return cudaErrorNotSupported;
  if constexpr (MMA) {
    const long long rows = static_cast<long long>(p.num_phys_pages) * p.num_kv_heads * S;
    bool wk = false, wv = false;
    if (!make_kv_tmap(&a.tmk, a.k_pool, p.kv_dtype, rows, D, S, &wk) ||
        !make_kv_tmap(&a.tmv, a.v_pool, p.kv_dtype, rows, D, S, &wv) || wk != wv)
      return cudaErrorNotSupported;
    a.whole_page = wk ? 1 : 0;
  }
  auto kern = k_sched<T, TQ, D, G, SEL>;
  cudaError_t e = ensure_smem(kern, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess ||
      per_sm < 1)
    return cudaErrorNotSupported;
  const int capacity = device_sm_count() * per_sm;
  const int units = p.batch * p.num_kv_heads;

  // Cost model of the split (SALS, AICPU Tiling: tasks planned from the
  // shapes before the compute).  Upper bounds from the page table's width:
  //  - scan time ~ every unit's candidate metadata at the planning bandwidth;
  //  - selection time of one unit ~ a fixed part plus a part per key;
  //  - selectors ~ enough that the units' selections keep up with the scan.
  const double bw = 6.0e12;
  const int cand = std::max(0, p.max_pages_per_seq - p.n_sink_pages - p.n_recent_pages);
  const double t_scan = static_cast<double>(units) * cand * rb / bw;
  const double t_sel = 1.5e-6 + cand * 0.8e-9 + (SEL == 1 ? 1.0e-6 : 0.0);
  // a unit's selection takes several microseconds of mostly latency: one
  // selector per unit where a quarter of the GPU's slots allow it, else as
  // many as keep up with the scan
  int n_selectors = units;
  if (units > capacity / 4)
    n_selectors = std::max(capacity / 4, static_cast<int>(std::ceil(units * t_sel / std::max(t_scan, 1.0e-6))));
  n_selectors = std::max(1, std::min(n_selectors, std::min(units, std::max(1, capacity / 2))));
  // attend task size: about two tasks per worker in all, at most kMaxSplits
  // tasks (partials) per unit
  const int att_pages = std::min(n_sel, p.max_pages_per_seq);
  const double ppt_target = static_cast<double>(units) * att_pages / (2.0 * std::max(capacity - n_selectors, 1));
  int spw = static_cast<int>(std::lround(ppt_target / (kConsumerWarps * pps)));
  spw = std::max(stages / kConsumerWarps, std::min(spw, 4));  // every slot of a warp used
  while ((att_pages + kConsumerWarps * spw * pps - 1) / (kConsumerWarps * spw * pps) > kMaxSplits) ++spw;
  if (spw > 64) return cudaErrorNotSupported;

  a.R = R;
  a.PPS = pps;
  a.SPW = spw;
  a.stages = stages;
  a.n_selectors = n_selectors;
  a.stage_bytes = sb;
  a.row_bytes = rb;
  a.page_bytes = pb;
  a.qbytes = qbytes;
  a.off_qbuf = static_cast<uint32_t>(off_qbuf);
  a.off_merge = static_cast<uint32_t>(off_merge);
  a.off_spt = static_cast<uint32_t>(off_spt);
  a.off_ssel = static_cast<uint32_t>(off_ssel);
  a.off_topk = static_cast<uint32_t>(off_topk);
  a.off_sP = static_cast<uint32_t>(off_sP);
  a.off_sqbar = static_cast<uint32_t>(off_sqbar);
  a.off_tps = static_cast<uint32_t>(off_tps);
  a.off_fixed = static_cast<uint32_t>(off_fixed);
  a.pt_cached = p.max_pages_per_seq % 4 == 0 ? 1 : 0;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(capacity);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, typename TQ, int SEL>
cudaError_t sched_dispatch(const spg_params& p, const SchedArgs& a, cudaStream_t st) {
  const int G = p.num_q_heads / p.num_kv_heads;
#define SPG_SC(D_, G_) \
  if (p.head_dim == D_ && G == G_) return sched_typed<T, TQ, D_, G_, SEL>(p, a, st);
  SPG_SC(128, 1) SPG_SC(128, 2) SPG_SC(128, 4) SPG_SC(128, 8)
  SPG_SC(64, 1) SPG_SC(64, 2) SPG_SC(64, 4) SPG_SC(64, 8)
#undef SPG_SC
  return cudaErrorNotSupported;
}

}  // namespace

bool sched_supported(const spg_params& p, int append) {
  if (p.selector != SPG_SEL_QUEST && p.selector != SPG_SEL_SKETCH_INT4) return false;
  if (p.max_pages_per_seq > kSchedMaxPages || p.batch > kSchedMaxBatch) return false;
  if (p.selector == SPG_SEL_SKETCH_INT4 && (p.page_size > 128 || p.sketch_dim != 16)) return false;
  if (append && p.n_recent_pages < 1) return false;  // the appended token's page must be forced
  return true;
}

cudaError_t launch_sched(const spg_params& p, const void* q, const void* k_pool,
                         const void* v_pool, const void* k_scale, const void* v_scale,
                         const int32_t* page_table, const int32_t* seq_lens, void* minmax,
                         const uint8_t* sketch, const float* sketch_scale, const float* proj,
                         int32_t* sel, int32_t* sel_cnt, float* out, float* lse, int append,
                         const Workspace& ws, cudaStream_t stream) {
  SchedArgs a{};
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.k_scale = static_cast<const __half*>(k_scale);
  a.v_scale = static_cast<const __half*>(v_scale);
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.minmax = minmax;
  // written only by the append (sparse_decode_step owns writable metadata)
  a.sketch = const_cast<uint8_t*>(sketch);
  a.sketch_scale = const_cast<float*>(sketch_scale);
  a.proj = proj;
  a.sel = sel;
  a.sel_cnt = sel_cnt;
  a.out = out;
  a.lse = lse;
  a.err = ws.err;
  a.ctr = ws.sched_ctr;
  a.uflags = ws.sched_flags;
  a.keys = reinterpret_cast<uint32_t*>(ws.scores);
  a.slices = ws.slices;
  a.iq = ws.iq;
  a.pm = ws.pm;
  a.pl = ws.pl;
  a.pacc = ws.pacc;
  a.B = p.batch;
  a.Hkv = p.num_kv_heads;
  a.S = p.page_size;
  a.MP = p.max_pages_per_seq;
  a.n_phys = p.num_phys_pages;
  a.n_sink = p.n_sink_pages;
  a.n_recent = p.n_recent_pages;
  a.n_sel = n_sel_pages(p);
  a.append = append;
  a.units = p.batch * p.num_kv_heads;
  const float scale = p.softmax_scale > 0.f ? p.softmax_scale
                                            : 1.0f / sqrtf(static_cast<float>(p.head_dim));
  a.scale_log2 = scale * kLog2e;
  a.inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(p.head_dim));
  a.top_p = p.top_p;
  a.min_pages = p.min_pages;
  a.tau = p.selector == SPG_SEL_SKETCH_INT4 ? 1.0f : scale;
  if (p.selector == SPG_SEL_QUEST) {
    switch (p.kv_dtype) {
      case SPG_F16:
        return sched_dispatch<__half, __half, 0>(p, a, stream);
      case SPG_BF16:
        return sched_dispatch<__nv_bfloat16, __nv_bfloat16, 0>(p, a, stream);
      default:
        if (p.q_dtype == SPG_F16) return sched_dispatch<int8_t, __half, 0>(p, a, stream);
        return sched_dispatch<int8_t, __nv_bfloat16, 0>(p, a, stream);
    }
  }
  switch (p.kv_dtype) {
    case SPG_F16:
      return sched_dispatch<__half, __half, 1>(p, a, stream);
    case SPG_BF16:
      return sched_dispatch<__nv_bfloat16, __nv_bfloat16, 1>(p, a, stream);
    default:
      if (p.q_dtype == SPG_F16) return sched_dispatch<int8_t, __half, 1>(p, a, stream);
      return sched_dispatch<int8_t, __nv_bfloat16, 1>(p, a, stream);
  }
}

}  // namespace spg
