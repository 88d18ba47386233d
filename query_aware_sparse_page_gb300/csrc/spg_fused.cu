// The whole decode step in one launch: metadata append (Quest), page scoring,
// exact top-k, sparse flash-decoding and the log-sum-exp merge, with one
// thread-block cluster of up to 8 CTAs per (batch, kv-head) unit.
//
// Sources: Quest 完全拆解 (关键性估计算法: insert-time min/max, 核心机制: the
// per-page bound, 三段式 kernel: estimate -> top-k -> approximate attention);
// SALS长序列推理优化 (QSI scoring and exact top-k, SFAA attention, AICPU
// Tiling challenge 2: a row split across cores merged by a reduction);
// SequenceO1 close reading §2.4 / §3.3 (fusing selection and attention: the
// indices never leave the chip here, they cross shared memory).
//
// Phases of one cluster (every CTA has 4 consumer warps, 1 producer warp and
// 1 auxiliary warp; each ring stage has one owner warp, stage k belonging to
// warp k % 4):
//  1. scan: the unit's candidate pages are split into contiguous chunks, one
//     per CTA.  Metadata is stored per sequence in logical page order, so a
//     chunk's rows (Quest: m and M, 2*d elements; sketch: the block's int4
//     codes) are one contiguous range; the producer streams it into the
//     shared-memory ring with one cp.async.bulk per stage of up to 64 rows.
//     Quest rows are scored 16 pages per tensor-core tile (A = the rows,
//     B = [q-; q+] for the group's query rows); sketch blocks one per lane
//     by int4 x int8 dots and a log-sum-exp.  Each order-preserving key goes
//     straight into the leader CTA's shared memory (st.shared::cluster), and
//     each warp reports its keys' min / max.
//  2. cluster barrier; the leader (rank 0) runs the exact top-k over the
//     keys, adds the forced pages, writes sel / sel_cnt, and pushes each
//     CTA's slice of the selection (physical page, valid tokens) into that
//     CTA's shared memory with asynchronous stores (st.async) that complete
//     the bytes of an mbarrier in the receiving CTA, plus one remote arrive
//     carrying the byte count; each CTA starts attending as soon as its own
//     slice has landed (no cluster barrier).
//  3. attend: each consumer warp copies the K/V pages of its own ring stages
//     (fp16/bf16, and int8 with d = 128 and an fp16 query: one 3-D TMA copy
//     per page for K and for V, landing as 128-byte-swizzled tiles for the
//     tensor-core consumers; other int8 shapes: bulk copies for the CUDA-core
//     consumer; int8 scales by bulk copy) and refills a stage as soon as it
//     has consumed it; the CTA's partial (m, l, acc) per query row goes into
//     the leader's shared memory.
//     The partials land where the leader kept its keys: a CTA writes them
//     only after the leader's auxiliary warp has signalled, with a release
//     at cluster scope made after the leader's last read of its keys.
//  4. cluster barrier; the leader merges the partials and writes out / lse.
// An auxiliary warp of the last CTA applies the metadata append of the new
// token during the scan (Quest min/max of its page; the sketch of a block it
// completes, split over every CTA's auxiliary warp, and its producer warp
// when that has nothing left to wait for): that page is forced, so nothing
// in the step reads it.  The leader's auxiliary warp bulk-copies the unit's
// page-table row into shared memory when it fits.
// Every thread arrives (relaxed) on the cluster barrier as it starts and
// waits before its warp's first access to another CTA's shared memory, so
// every CTA has started before it is written to.  Beyond that, CTAs wait on
// one another only at the cluster barriers after the scan and before the
// merge, which every thread of every CTA reaches on every path, and for the
// slice and the keys-free signal the leader sends; all mbarrier waits are
// bounded (SPG_DEVERR_TIMEOUT) and a CTA whose waits run out still reaches
// the cluster barriers.
#include "spg_append.cuh"
#include "spg_attn_core.cuh"
#include "spg_internal.h"
#include "spg_select_core.cuh"

namespace spg {
namespace {

constexpr int kMaxCluster = 8;
constexpr int kMaxScanRows = 64;
constexpr int kMaxPagesPerStage = 8;
constexpr int kFusedMaxPages = 8192;  // candidate keys the leader holds
// A stage carries several pages (or metadata rows): the handshake of a ring
// stage costs about the same whatever its size, so ~16 KB stages and a
// 64 KB ring per CTA (two CTAs per SM) keep HBM busy where one page per
// stage would not.
constexpr int kStageBytesTarget = 16 * 1024;
constexpr int kRingBytesTarget = 64 * 1024;

struct FusedArgs {
  CUtensorMap tmk, tmv;  // K / V pools as page tiles (fp16/bf16 pools)
  int whole_page;        // the maps are 3-D: one copy per page
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const __half* k_scale;
  const __half* v_scale;
  const int32_t* page_table;
  const int32_t* seq_lens;
  void* minmax;  // written only by the append
  const uint8_t* sketch;
  const float* sketch_scale;
  uint8_t* sketch_w;       // the same arrays, written only by the append
  float* sketch_scale_w;
  const float* proj;
  int32_t* sel;
  int32_t* sel_cnt;
  float* out;
  float* lse;
  int32_t* err;
  int Hkv, S, MP, n_phys, n_sink, n_recent, n_sel, stages, rows_per_stage, append;
  float top_p, tau;  // adaptive budget (top_p 0: off)
  int min_pages;
  int cluster, pages_per_stage;
  uint32_t stage_bytes, row_bytes, page_bytes, ring_bytes, keys_off, sel_off, att_off;
  uint32_t pt_off;  // leader: the unit's page-table row, when it fits (0: not cached)
  float scale_log2, inv_sqrt_d;
};

// consumer-only barrier (named barrier 1, the 4 consumer warps)
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

template <typename T, int CPL>
__device__ __forceinline__ void smem_chunk(const uint8_t* p, uint32_t (&w)[CPL / 2]) {
  if constexpr (CPL == 8) {
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
  } else {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    w[0] = r.x; w[1] = r.y;
  }
}

// Sketch of the block completed by the token at L-1 (when L is a multiple of
// S; SALS长序列推理优化, the low-rank index key of a block), split over the
// cluster's C CTAs: CTA r takes tokens [r*S/C, (r+1)*S/C), one token per
// lane.  Its auxiliary warp computes all DS = 16 sketch dimensions, or, when
// the CTA's scan fits its ring (the producer warp then has nothing left to
// wait for), dimensions 0-7 while the producer warp computes 8-15.  Keys are
// dequantised (int8 code times its fp16 scale, exact in fp32) and projected
// in fp32 with each product rounded and each dimension's sum taken in
// channel order (no fused multiply-add), so the split does not change a
// value.  Part 1 (during the scan) keeps the lane's values in registers and
// sends the CTA's |max| to every CTA; part 2 (after the scan barrier) forms
// the block scale absmax / 7 and writes codes rint(v / scale) clamped to
// [-7, 7], two per byte.  The block is the tail block of this step (forced,
// never scored), so nothing in the step reads what is written.
constexpr int kSketchVals = 16;  // one token's 16 sketch values per lane: S / C <= 32

// half: 0 = the auxiliary warp, 1 = the producer warp (split only); every
// lane of both warps calls it when split (they meet at named barrier 2)
template <typename T, int D>
__device__ void sketch_append_part1(const FusedArgs& a, int b, int h, int L, int lane, uint32_t rank,
                                    int C, int half, bool split, float (&v)[kSketchVals],
                                    float* s_samax, float* s_hmax) {
  constexpr int DS = 16;
  const int S = a.S, blk = L / S - 1, tpc = S / C;
  const int t = static_cast<int>(rank) * tpc + lane;  // this lane's token
  const int phys = a.page_table[static_cast<size_t>(b) * a.MP + blk];
  float amax = 0.f;
#pragma unroll
  for (int u = 0; u < DS; ++u) v[u] = 0.f;
  if (phys >= 0 && phys < a.n_phys) {
    if (lane < tpc) {
      const size_t ph = static_cast<size_t>(phys) * a.Hkv + h;
      float sc = 1.f;
      if constexpr (is_i8<T>()) sc = __half2float(a.k_scale[ph * S + t]);
      const T* krow = static_cast<const T*>(a.k_pool) + (ph * S + t) * D;
      if (split) {
        float w[DS / 2];
        sketch_project_row_part<T, D, DS / 2>(krow, sc, a.proj, half * (DS / 2), w);
#pragma unroll
        for (int u = 0; u < DS / 2; ++u) {
          v[u] = w[u];
          amax = fmaxf(amax, fabsf(w[u]));
        }
      } else {
        sketch_project_row<T, D>(krow, sc, a.proj, v);
#pragma unroll
        for (int u = 0; u < DS; ++u) amax = fmaxf(amax, fabsf(v[u]));
      }
    }
  } else if (lane == 0 && rank == 0 && half == 0) {
    record_error(a.err, SPG_DEVERR_PAGE_ID);
  }
  amax = warp_max(amax);
  if (split) {
    // the two warps' |max| (named barrier 2: the producer and auxiliary warps)
    if (lane == 0) s_hmax[half] = amax;
    asm volatile("bar.sync 2, 64;" ::: "memory");
    amax = fmaxf(s_hmax[0], s_hmax[1]);
    if (half != 0) return;
  }
  // every CTA needs every CTA's |max| after the scan barrier
  if (lane < C) st_cluster_f32(map_rank(s_samax + rank, static_cast<uint32_t>(lane)), amax);
}

template <typename T, int D>
__device__ void sketch_append_part2(const FusedArgs& a, int b, int h, int L, int lane, uint32_t rank,
                                    int C, int half, bool split, const float (&v)[kSketchVals],
                                    const float* s_samax) {
  constexpr int DS = 16;
  const int S = a.S, blk = L / S - 1, tpc = S / C;
  const int t = static_cast<int>(rank) * tpc + lane;
  const int phys = a.page_table[static_cast<size_t>(b) * a.MP + blk];
  if (phys < 0 || phys >= a.n_phys) return;
  float amax = 0.f;
  for (int r = 0; r < C; ++r) amax = fmaxf(amax, s_samax[r]);
  const float scale = amax > 0.f ? __fdiv_rn(amax, 7.0f) : 1.0f;
  const size_t lrow = (static_cast<size_t>(b) * a.Hkv + h) * a.MP + blk;
  auto code2 = [&](float x0, float x1) {
    const int c0 = max(-7, min(7, static_cast<int>(rintf(__fdiv_rn(x0, scale)))));
    const int c1 = max(-7, min(7, static_cast<int>(rintf(__fdiv_rn(x1, scale)))));
    return static_cast<uint32_t>((c0 & 0xf) | ((c1 & 0xf) << 4));
  };
  if (lane < tpc) {
    uint8_t* dst = a.sketch_w + (lrow * S + t) * (DS / 2);
    if (split) {  // this warp's half of the token's 8 bytes
      uint32_t w = 0u;
#pragma unroll
      for (int k = 0; k < DS / 4; ++k) w |= code2(v[2 * k], v[2 * k + 1]) << (8 * k);
      *reinterpret_cast<uint32_t*>(dst + 4 * half) = w;
    } else {
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int k = 0; k < DS / 2; ++k) w[k >> 2] |= code2(v[2 * k], v[2 * k + 1]) << (8 * (k & 3));
      *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    }
  }
  if (rank == 0 && lane == 0 && half == 0) a.sketch_scale_w[lrow] = scale;
}

template <typename T, typename TQ, int D, int G, int SEL>
__global__ void __launch_bounds__((kConsumerWarps + 2) * 32)
    k_fused(const __grid_constant__ FusedArgs a) {
  constexpr int CW = kConsumerWarps;
  // consumer: 1 = tensor cores on fp16/bf16 pages, 2 = tensor cores on int8
  // pages (D = 128, fp16 query), 0 = CUDA cores; 1 and 2 take TMA tiles
  constexpr int CONS = !is_i8<T>() ? 1 : ((D == 128 && std::is_same<TQ, __half>::value) ? 2 : 0);
  constexpr bool MMA = CONS != 0;
  // Quest metadata type: the pool's, or the query's for int8 pools
  using TM = std::conditional_t<is_i8<T>(), TQ, T>;
  const int C = a.cluster;
  using Consumer = std::conditional_t<
      CONS == 1, AttnMma<T, D, G>,
      std::conditional_t<CONS == 2, AttnMmaI8<G>, AttnConsumer<T, D, G, 1>>>;

  extern __shared__ __align__(128) uint8_t smem_raw[];
  // TMA tiles with 128-byte swizzle want 1024-byte aligned destinations
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ float s_qbar[SEL ? 256 : 1];
  __shared__ float s_P[SEL ? 256 * 16 : 1];
  __shared__ int s_qc[4];
  __shared__ float s_sq;
  __shared__ __align__(8) uint64_t s_ptbar;  // leader: the page-table row has landed
  __shared__ __align__(8) uint64_t s_slice;  // non-leader: its slice of the selection has landed
  __shared__ __align__(8) uint64_t s_kfree;  // non-leader: the leader no longer reads its keys
  __shared__ int s_natt;  // pages of the selection this CTA attends to
  __shared__ float s_samax[kMaxCluster];  // sketch append: each CTA's |max|
  __shared__ float s_hmax[2];             // sketch append: the two warps' |max| (split)
  float sk_v[SEL ? kSketchVals : 1];       // sketch append: this lane's projected values

  const int S = a.S, STAGES = a.stages, R = a.rows_per_stage, PPS = a.pages_per_stage;
  const uint32_t sbytes = a.stage_bytes, rb = a.row_bytes, pbytes = a.page_bytes;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.ring_bytes);
  uint64_t* empty = full + kMaxStages;
  int* s_np = reinterpret_cast<int*>(empty + kMaxStages);                // [stages] pages in stage
  int* s_nv = s_np + kMaxStages;                                          // [stages][8] valid tokens
  uint32_t* s_keys = reinterpret_cast<uint32_t*>(smem + a.keys_off);       // leader: keys
  float* s_part = reinterpret_cast<float*>(smem + a.keys_off);            // leader: partials
  int* s_sel = reinterpret_cast<int*>(smem + a.sel_off);                  // leader: selection
  TopkShared& tk = *reinterpret_cast<TopkShared*>(ring);  // leader: top-k state (ring idle then)
  uint32_t* s_mm = reinterpret_cast<uint32_t*>(smem + a.att_off);         // leader: [2][C*CW] key min/max
  int* s_att_ph = reinterpret_cast<int*>(s_mm + 2 * kMaxCluster * CW);    // [n_sel] physical pages
  int* s_att_nv = s_att_ph + a.n_sel;                                     // [n_sel] valid tokens
  int* s_pt = reinterpret_cast<int*>(smem + a.pt_off);                    // leader: page-table row

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int unit = blockIdx.y;
  const int Hkv = a.Hkv, b = unit / Hkv, h = unit % Hkv, Hq = Hkv * G;

  // every stage has one owner: scan stage / attention stage k belongs to
  // consumer warp k % CW (STAGES is a multiple of CW, so a ring slot always
  // has the same owner)
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&s_ptbar, 1);
    mbar_init(&s_slice, 1);
    mbar_init(&s_kfree, 1);
    mbar_fence_init();
  }
  if constexpr (MMA) {
    if (threadIdx.x == CW * 32) {
      tma_prefetch_desc(&a.tmk);
      tma_prefetch_desc(&a.tmv);
    }
  }
  // every CTA of the cluster must have started before another touches its
  // shared memory: arrive now, wait before the first remote access below
  cluster_arrive_relaxed();
  pdl_wait();
  int L = a.seq_lens[b];
  if (L < 0 || L > a.MP * S) {
    if (rank == 0 && threadIdx.x == 0) record_error(a.err, SPG_DEVERR_SEQ_LEN);
    L = 0;
  }
  const int P = (L + S - 1) / S;
  const int lo = min(a.n_sink, P), hi = max(P - a.n_recent, lo), nc = hi - lo;
  __syncthreads();

  // ------------------------------------------------------------------ scan
  const int cpc = (nc + C - 1) / C;
  const int c0 = lo + min(nc, static_cast<int>(rank) * cpc);
  const int rows = lo + min(nc, static_cast<int>(rank + 1) * cpc) - c0;
  const int n_scan = (rows + R - 1) / R;
  // the sketch append of a completed block: split between the auxiliary and
  // producer warps when the producer issues every scan stage without waiting
  const bool sk_append = SEL == 1 && a.append && L > 0 && L % S == 0;
  const bool sk_split = sk_append && n_scan <= STAGES;
  const uint32_t keys_leader = map_rank(s_keys, 0);
  const uint32_t mm_leader = map_rank(s_mm, 0);
  bool ok = true;

  if (warp == CW) {
    if (a.pt_off == 0 && rank == C - 1 && lane == 0 && P > 0) {
      // the attend phase looks the selected pages up in this row: have it in
      // L2 by then
      const int32_t* pt = a.page_table + static_cast<size_t>(b) * a.MP;
      const uint32_t bytes = (static_cast<uint32_t>(P) * 4u) & ~15u;  // within the row
      if ((reinterpret_cast<uintptr_t>(pt) & 15u) == 0 && bytes > 0) bulk_prefetch_l2(pt, bytes);
    }
    // producer: metadata is stored in logical page order, so this CTA's rows
    // are one contiguous range: one bulk copy per stage of R rows
    const size_t lrow0 = static_cast<size_t>(unit) * a.MP + c0;
    const uint8_t* src0 = SEL == 0 ? static_cast<const uint8_t*>(a.minmax) + lrow0 * rb
                                   : a.sketch + lrow0 * rb;
    for (int k = 0; k < n_scan; ++k) {
      const int stage = k % STAGES, nr = min(R, rows - k * R);
      bool lok = true;
      if (lane == 0 && k >= STAGES) lok = mbar_wait_bounded(&empty[stage], ((k / STAGES) - 1) & 1);
      ok = __shfl_sync(0xffffffffu, lok ? 1 : 0, 0) != 0;
      if (!ok) {
        if (lane == 0) record_error(a.err, SPG_DEVERR_TIMEOUT);
        break;
      }
      if (lane == 0) {
        mbar_expect_tx(&full[stage], nr * rb);
        bulk_g2s(ring + static_cast<size_t>(stage) * sbytes, src0 + static_cast<size_t>(k) * R * rb,
                 nr * rb, &full[stage]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[stage]);
    }
    cluster_wait();
    if constexpr (SEL == 1)  // the producer's half of the sketch append
      if (sk_split)
        sketch_append_part1<T, D>(a, b, h, L, lane, rank, C, 1, true, sk_v, s_samax, s_hmax);
  } else if (warp == CW + 1) {
    // auxiliary warp: the metadata append of the token at L-1.  Its page is
    // forced (n_recent >= 1), so neither this step's scan nor its attend
    // reads that metadata; done here it overlaps the scan.
    if (a.pt_off != 0 && rank == 0 && lane == 0) {
      // the leader looks the selected pages up in this row: one bulk copy of
      // its first P entries (rounded up to 16 bytes, within the row: the
      // host caches only rows of a multiple of 4 entries) lands it in shared
      // memory during the scan
      const uint32_t bytes = (static_cast<uint32_t>(P) * 4u + 15u) & ~15u;
      if (bytes > 0) {
        mbar_expect_tx(&s_ptbar, bytes);
        bulk_g2s(s_pt, a.page_table + static_cast<size_t>(b) * a.MP, bytes, &s_ptbar);
      }
      mbar_arrive(&s_ptbar);
    }
    if constexpr (SEL == 0) {
      if (a.append && rank == C - 1 && L > 0) {
        if constexpr (is_i8<T>())
          minmax_append_warp_i8<TM, D>(static_cast<const int8_t*>(a.k_pool), a.k_scale, a.page_table,
                                       static_cast<TM*>(a.minmax), a.err, a.Hkv, a.S, a.MP, a.n_phys,
                                       b, h, L, lane);
        else
          minmax_append_warp<T, D>(static_cast<const T*>(a.k_pool), a.page_table,
                                   static_cast<T*>(a.minmax), a.err, a.Hkv, a.S, a.MP, a.n_phys, b, h,
                                   L, lane);
      }
    }
    cluster_wait();
    if constexpr (SEL == 1) {
      // the sketch of a block is written when the block fills (every CTA's
      // aux warp takes a slice)
      if (sk_append)
        sketch_append_part1<T, D>(a, b, h, L, lane, rank, C, 0, sk_split, sk_v, s_samax, s_hmax);
    }
  } else {
    // consumers
    uint32_t kmn = 0xffffffffu, kmx = 0u;  // of the keys this warp produces
    if constexpr (SEL == 0) {
      QuestMma<TM, D, G> qm;
      qm.init(static_cast<const TM*>(a.q) + (static_cast<size_t>(b) * Hq + h * G) * D, lane);
      cluster_wait();  // (the first stage is in flight meanwhile)
      for (int ks = warp; ks < n_scan; ks += CW) {
        const int stage = ks % STAGES;
        if (!mbar_wait_bounded(&full[stage], (ks / STAGES) & 1)) {
          if (lane == 0) record_error(a.err, SPG_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        const int nr = min(R, rows - ks * R);
        const TM* st = reinterpret_cast<const TM*>(ring + static_cast<size_t>(stage) * sbytes);
        for (int ti = 0; ti * 16 < nr; ++ti) {  // the stage's 16-page tiles
          const int pt0 = c0 + ks * R + ti * 16;
          float s0, s1;
          qm.tile(st + ti * 16 * 2 * D, pt0, lane, s0, s1);
          if ((lane & 3) == 0) {
            const int g = lane >> 2;
            if (ti * 16 + g < nr) {
              const uint32_t k0 = score_key(s0);
              st_cluster_u32(keys_leader + 4u * (pt0 + g - lo), k0);
              kmn = min(kmn, k0);
              kmx = max(kmx, k0);
            }
            if (ti * 16 + g + 8 < nr) {
              const uint32_t k1 = score_key(s1);
              st_cluster_u32(keys_leader + 4u * (pt0 + g + 8 - lo), k1);
              kmn = min(kmn, k1);
              kmx = max(kmx, k1);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
      }
    } else {
      // index query of the group, built by the consumer warps only
      const TQ* qb = static_cast<const TQ*>(a.q) + (static_cast<size_t>(b) * Hq + h * G) * D;
      constexpr int DS = 16;
      {  // P (16-byte aligned): all of a thread's loads in flight at once
        constexpr int NV = D * DS / 4 / (CW * 32);
        const float4* P4 = reinterpret_cast<const float4*>(a.proj);
        float4 v[NV];
#pragma unroll
        for (int u = 0; u < NV; ++u) v[u] = __ldg(P4 + threadIdx.x + u * CW * 32);
#pragma unroll
        for (int u = 0; u < NV; ++u) reinterpret_cast<float4*>(s_P)[threadIdx.x + u * CW * 32] = v[u];
      }
      consumers_sync();
      if (warp == 0) {
        int c4[4];
        float sqv;
        sketch_index_query_warp<TQ>(qb, G, D, s_P, s_qbar, lane, c4, sqv);
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) s_qc[k] = c4[k];
          s_sq = sqv;
        }
      }
      consumers_sync();
      const int qc[4] = {s_qc[0], s_qc[1], s_qc[2], s_qc[3]};
      const int qbias = sketch_query_bias(qc);
      const float sq = s_sq;
      cluster_wait();
      const size_t lrow0 = static_cast<size_t>(unit) * a.MP + c0;
      for (int ks = warp; ks < n_scan; ks += CW) {
        const int stage = ks % STAGES;
        const int nr = min(R, rows - ks * R);
        // the lane's block scale, loaded while the stage's codes land
        const float bsc = lane < nr ? __ldg(a.sketch_scale + lrow0 + ks * R + lane) : 0.f;
        if (!mbar_wait_bounded(&full[stage], (ks / STAGES) & 1)) {
          if (lane == 0) record_error(a.err, SPG_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        const uint8_t* st = ring + static_cast<size_t>(stage) * sbytes;
        // the stage's blocks (nr <= 32), one per lane; every scored block is
        // full (the open tail block is forced, never scored)
        if (lane < nr) {
          const float cz = __fmul_rn(__fmul_rn(sq, bsc), a.inv_sqrt_d);
          const float sc = sketch_block_score_lane(st + lane * rb, S, qc, qbias, cz);
          const uint32_t k0 = score_key(sc);
          st_cluster_u32(keys_leader + 4u * (c0 + ks * R + lane - lo), k0);
          kmn = min(kmn, k0);
          kmx = max(kmx, k0);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
      }
    }
    kmn = __reduce_min_sync(0xffffffffu, kmn);
    kmx = __reduce_max_sync(0xffffffffu, kmx);
    if (lane == 0) {
      st_cluster_u32(mm_leader + 4u * (rank * CW + warp), kmn);
      st_cluster_u32(mm_leader + 4u * (kMaxCluster * CW + rank * CW + warp), kmx);
    }
  }
  cluster_sync();  // every key (and every warp's key min / max) is in the leader

  if constexpr (SEL == 1) {
    if (warp == CW + 1 && sk_append)
      sketch_append_part2<T, D>(a, b, h, L, lane, rank, C, 0, sk_split, sk_v, s_samax);
    else if (warp == CW && sk_split)
      sketch_append_part2<T, D>(a, b, h, L, lane, rank, C, 1, true, sk_v, s_samax);
  }

  // ------------------------------------------------------------- selection
  if (rank == 0) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int nf = P - nc;
    int k_top = min(max(a.n_sel - nf, 0), nc);
    for (int i = tid; i < lo; i += nt) s_sel[i] = i;
    if (k_top == nc) {
      for (int i = tid; i < nc; i += nt) s_sel[lo + i] = lo + i;
    } else if (k_top > 0) {
      for (int i = tid; i < 512; i += nt) reinterpret_cast<int4*>(tk.hist)[i] = make_int4(0, 0, 0, 0);
      if (warp == 0) {  // the keys' min / max, from the scanning warps' reports
        uint32_t kn = lane < C * CW ? s_mm[lane] : 0xffffffffu;
        uint32_t kx = lane < C * CW ? s_mm[kMaxCluster * CW + lane] : 0u;
        kn = __reduce_min_sync(0xffffffffu, kn);
        kx = __reduce_max_sync(0xffffffffu, kx);
        if (lane == 0) {
          tk.kmin = kn;
          tk.kmax = kx;
        }
      }
      __syncthreads();
      block_topk(s_keys, nc, k_top, lo, s_sel + lo, tk, true, true);
    }
    if (a.top_p > 0.f && k_top > 0) {
      // the adaptive budget trims the chosen candidates (the ring is idle:
      // its scratch follows the top-k state)
      __syncthreads();
      uint32_t* tps = reinterpret_cast<uint32_t*>(ring + ((sizeof(TopkShared) + 127) & ~size_t(127)));
      k_top = topp_trim(s_keys, nc, s_sel + lo, k_top, lo, a.tau, a.top_p, a.min_pages, tps,
                        reinterpret_cast<int*>(tps + kTopPScratchWords),
                        reinterpret_cast<float*>(tps + kTopPScratchWords + 40));
    }
    __syncthreads();
    for (int j = tid; j < P - hi; j += nt) s_sel[lo + k_top + j] = hi + j;
    const int count = lo + k_top + (P - hi);
    __syncthreads();
    if (a.pt_off != 0 && !mbar_wait_bounded(&s_ptbar, 0) && tid == 0)
      record_error(a.err, SPG_DEVERR_TIMEOUT);
    // the selection to HBM, and each CTA's slice of it (physical page, valid
    // tokens) into that CTA's shared memory, so that its attend phase starts
    // from local data
    int32_t* gsel = a.sel + static_cast<size_t>(unit) * a.n_sel;
    const int ppc = (count + C - 1) / C;
    for (int i = tid; i < a.n_sel; i += nt) {
      const int lp = i < count ? s_sel[i] : -1;
      gsel[i] = lp;
      if (i < count) {
        int ph = -1, nv = 0;
        if (lp < 0 || lp >= P) {
          record_error(a.err, SPG_DEVERR_SEL);
        } else {
          ph = a.pt_off != 0 ? s_pt[lp] : a.page_table[static_cast<size_t>(b) * a.MP + lp];
          if (ph < 0 || ph >= a.n_phys) {
            record_error(a.err, SPG_DEVERR_PAGE_ID);
            ph = -1;
          } else {
            nv = min(S, L - lp * S);
          }
        }
        const uint32_t r = static_cast<uint32_t>(i / ppc), j = static_cast<uint32_t>(i - r * ppc);
        if (r == 0) {
          s_att_ph[j] = ph;
          s_att_nv[j] = nv;
        } else {
          const uint32_t bar = map_rank(&s_slice, r);
          st_async_u32(map_rank(s_att_ph + j, r), static_cast<uint32_t>(ph), bar);
          st_async_u32(map_rank(s_att_nv + j, r), static_cast<uint32_t>(nv), bar);
        }
      }
    }
    if (tid < C) {
      const int na = min(count, (tid + 1) * ppc) - min(count, tid * ppc);
      if (tid == 0) {
        s_natt = na;
      } else {
        // the slice's bytes: na (ph, nv) pairs and na itself
        const uint32_t r = static_cast<uint32_t>(tid), bar = map_rank(&s_slice, r);
        st_async_u32(map_rank(&s_natt, r), static_cast<uint32_t>(na), bar);
        mbar_arrive_expect_tx_cluster(bar, 4u * (2u * static_cast<uint32_t>(na) + 1u));
      }
    }
    if (tid == 0) a.sel_cnt[unit] = count;
    __syncthreads();  // the leader's own slice
    // its keys are read no more: the other CTAs may write their partials
    // there (the auxiliary warp, idle from here on, takes the release's wait)
    if (warp == CW + 1 && lane > 0 && lane < C)
      mbar_arrive_cluster(map_rank(&s_kfree, static_cast<uint32_t>(lane)));
  } else {
    // wait for this CTA's slice (bounded); without it the CTA attends to nothing
    bool got = true;
    if (threadIdx.x == 0) {
      got = mbar_wait_bounded<true>(&s_slice, 0);
      if (!got) record_error(a.err, SPG_DEVERR_TIMEOUT);
    }
    if (__syncthreads_and(got ? 1 : 0) == 0 && threadIdx.x == 0) s_natt = 0;
    __syncthreads();
  }

  // ---------------------------------------------------------------- attend
  // Attend stage j holds pages [j * PPS, (j + 1) * PPS) of this CTA's slice;
  // stages are numbered on from the scan's (k = n_scan + j) and stage k
  // belongs to consumer warp k % CW, which issues its copies itself, keeps up
  // to STAGES / CW of its stages in flight and refills a slot as soon as it
  // has consumed it (a slot always has the same owner, so no handshake sits
  // between the consumer and the next copy into its slot).
  const int n_att = s_natt;
  Consumer cons;
  if (warp < CW) {
    cons.init(static_cast<const TQ*>(a.q) + (static_cast<size_t>(b) * Hq + h * G) * D,
              a.scale_log2, warp, lane);
    const uint32_t tile = static_cast<uint32_t>(S) * D * sizeof(T);
    const uint32_t scb = is_i8<T>() ? static_cast<uint32_t>(S) * 2 : 0u;
    const uint64_t pol = policy_evict_first();
    const int n_st = (n_att + PPS - 1) / PPS;
    auto issue = [&](int j) {
      const int k = n_scan + j, stage = k % STAGES;
      const int np = min(PPS, n_att - j * PPS);
      if (lane < np) {
        const int ph = s_att_ph[j * PPS + lane];
        uint8_t* dst = ring + static_cast<size_t>(stage) * sbytes + static_cast<size_t>(lane) * pbytes;
        s_nv[stage * kMaxPagesPerStage + lane] = ph >= 0 ? s_att_nv[j * PPS + lane] : 0;
        if (ph >= 0) {
          const size_t row = static_cast<size_t>(ph) * Hkv + h;
          mbar_expect_tx(&full[stage], 2 * tile + 2 * scb);
          if constexpr (MMA) {
            const int y = static_cast<int>(row) * S;
            if (a.whole_page) {
              tma_load_3d(dst, &a.tmk, 0, y, 0, &full[stage], pol);
              tma_load_3d(dst + tile, &a.tmv, 0, y, 0, &full[stage], pol);
            } else {
              // swizzled tiles of [S rows][128 bytes] for K, then for V
              constexpr int NT = D * static_cast<int>(sizeof(T)) / 128, EPT = 128 / sizeof(T);
#pragma unroll
              for (int hf = 0; hf < NT; ++hf) {
                tma_load_2d(dst + hf * S * 128, &a.tmk, hf * EPT, y, &full[stage], pol);
                tma_load_2d(dst + tile + hf * S * 128, &a.tmv, hf * EPT, y, &full[stage], pol);
              }
            }
          } else {
            bulk_g2s_hint(dst, static_cast<const T*>(a.k_pool) + row * S * D, tile, &full[stage], pol);
            bulk_g2s_hint(dst + tile, static_cast<const T*>(a.v_pool) + row * S * D, tile, &full[stage], pol);
          }
          if constexpr (is_i8<T>()) {
            bulk_g2s(dst + 2 * tile, a.k_scale + row * S, scb, &full[stage]);
            bulk_g2s(dst + 2 * tile + scb, a.v_scale + row * S, scb, &full[stage]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        s_np[stage] = np;
        mbar_arrive(&full[stage]);
      }
    };
    // this warp's slots last held scan stages it consumed (generic-proxy
    // reads) before the asynchronous copies that now land there
    fence_proxy_async();
    const int j0 = ((warp - n_scan) % CW + CW) % CW;
    int nxt = j0;  // the next of this warp's stages not yet issued
    for (int j = j0; ok && j < n_st; j += CW) {
      for (; nxt < n_st && nxt < j + STAGES; nxt += CW) issue(nxt);
      const int k = n_scan + j, stage = k % STAGES;
      if (!mbar_wait_bounded(&full[stage], (k / STAGES) & 1)) {
        ok = false;
        if (lane == 0) record_error(a.err, SPG_DEVERR_TIMEOUT);
        break;
      }
      const int np = s_np[stage];
      for (int i = 0; i < np; ++i) {
        const int nv = s_nv[stage * kMaxPagesPerStage + i];
        uint8_t* pg = ring + static_cast<size_t>(stage) * sbytes + static_cast<size_t>(i) * pbytes;
        if (nv > 0) {
          if constexpr (MMA)
            cons.consume(pg, S, nv, lane);
          else
            cons.consume(pg, S, nv);
        }
      }
      fence_proxy_async();  // reads (and zeroed slots) before the next copy into the slot
      __syncwarp();
    }
    if (!ok && lane == 0) {
      // wait (bounded) for the copies this warp may still have in flight
      for (int j = max(j0, nxt - STAGES); j < nxt; j += CW) {
        const int k = n_scan + j;
        mbar_wait_bounded(&full[k % STAGES], (k / STAGES) & 1);
      }
    }
    cons.fold();
  }
  pdl_trigger();

  // the CTA's partial (merge of its consumer warps) into the leader
  __syncthreads();
  float* s_m = reinterpret_cast<float*>(ring);  // [CW][G]
  float* s_l = s_m + CW * G;
  float* s_acc = s_l + CW * G;                   // [CW][G][D]
  if (warp < CW) cons.store(s_m, s_l, s_acc, lane);
  __syncthreads();
  const uint32_t part_leader = map_rank(s_part, 0);
  bool kfree = true;
  if (rank != 0) {
    // the partials go where the leader's keys were: wait for its signal
    // (long sent, normally); if that wait runs out the partial is not
    // written (the error is recorded)
    if (threadIdx.x == 0) {
      kfree = mbar_wait_bounded<true>(&s_kfree, 0);
      if (!kfree) record_error(a.err, SPG_DEVERR_TIMEOUT);
    }
    kfree = __syncthreads_and(kfree ? 1 : 0) != 0;
  }
  for (int idx = threadIdx.x; kfree && idx < G * D; idx += blockDim.x) {
    const int g = idx / D, c = idx % D;
    float M, Ls, A;
    lse_merge(s_m, s_l, s_acc, CW, G, D, g, c, M, Ls, A);
    // leader layout: m [C][G], l [C][G], acc [C][G][D]
    st_cluster_f32(part_leader + 4u * (C * G + C * G + (rank * G + g) * D + c), A);
    if (c == 0) {
      st_cluster_f32(part_leader + 4u * (rank * G + g), M);
      st_cluster_f32(part_leader + 4u * (C * G + rank * G + g), Ls);
    }
  }
  cluster_sync();  // every partial is in the leader

  if (rank == 0) {
    const float* pm = s_part;
    const float* pl = s_part + C * G;
    const float* pa = s_part + 2 * C * G;
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
      const int g = idx / D, c = idx % D;
      float M, Ls, A;
      lse_merge(pm, pl, pa, C, G, D, g, c, M, Ls, A);
      const size_t row = static_cast<size_t>(b) * Hq + h * G + g;
      a.out[row * D + c] = Ls > 0.f ? A / Ls : 0.f;
      if (c == 0 && a.lse) a.lse[row] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
    }
  }
}

template <typename T, typename TQ, int D, int G>
cudaError_t fused_typed(const spg_params& p, FusedArgs a, cudaStream_t st) {
  constexpr int threads = (kConsumerWarps + 2) * 32;  // + producer + auxiliary warp
  const int S = p.page_size;
  constexpr bool MMA = !is_i8<T>() || (D == 128 && std::is_same<TQ, __half>::value);
  // a page's K tile must start 1024-byte aligned for the swizzled TMA tiles
  const uint32_t pb = MMA ? (kv_stage_bytes<T, D>(S) + 1023u) & ~1023u : kv_stage_bytes<T, D>(S);
  using TM = std::conditional_t<is_i8<T>(), TQ, T>;  // Quest metadata type
  const uint32_t rb = p.selector == SPG_SEL_QUEST ? 2u * D * sizeof(TM) : static_cast<uint32_t>(S) * 8u;
  int pps = 1;
  while (pps * 2 <= kMaxPagesPerStage && (pps * 2) * pb <= static_cast<uint32_t>(kStageBytesTarget))
    pps *= 2;
  int R = static_cast<int>(std::max<uint32_t>(pps * pb, kStageBytesTarget) / rb);
  R = (min(R, kMaxScanRows) / 16) * 16;  // whole 16-page tensor-core tiles
  if (R < 16) return cudaErrorNotSupported;
  const uint32_t sb = std::max<uint32_t>(pps * pb, R * rb);
  // a multiple of the consumer warps: each ring slot has one owner
  int stages = max(32 / R, max(2, min(kMaxStages, static_cast<int>(kRingBytesTarget / sb))));
  stages = (stages + kConsumerWarps - 1) / kConsumerWarps * kConsumerWarps;
  if (stages > kMaxStages) return cudaErrorNotSupported;
  size_t ring = static_cast<size_t>(stages) * sb;
  ring = max(ring, sizeof(TopkShared));
  if (p.top_p > 0.f)  // the adaptive budget's scratch after the top-k state
    ring = max(ring, ((sizeof(TopkShared) + 127) & ~size_t(127)) + sizeof(uint32_t) * (kTopPScratchWords + 80));
  ring = max(ring, sizeof(float) * kConsumerWarps * G * (D + 2));
  ring = (ring + 127) & ~static_cast<size_t>(127);
  const size_t meta = sizeof(uint64_t) * 2 * kMaxStages +
                      sizeof(int) * (kMaxStages + kMaxStages * kMaxPagesPerStage);
  const size_t keys_off = (ring + meta + 127) & ~static_cast<size_t>(127);
  const size_t keys_bytes =
      max(sizeof(uint32_t) * p.max_pages_per_seq, sizeof(float) * kMaxCluster * G * (D + 2));
  const size_t sel_off = (keys_off + keys_bytes + 127) & ~static_cast<size_t>(127);
  const size_t att_off = (sel_off + sizeof(int) * n_sel_pages(p) + 127) & ~static_cast<size_t>(127);
  const size_t att_bytes = sizeof(uint32_t) * 2 * kMaxCluster * kConsumerWarps +
                           sizeof(int) * 2 * n_sel_pages(p);
  size_t smem = 1024 + att_off + att_bytes;  // + alignment slack
  if (smem > 227u * 1024u) return cudaErrorNotSupported;
  if constexpr (MMA) {
    const long long rows = static_cast<long long>(p.num_phys_pages) * p.num_kv_heads * S;
    bool wk = false, wv = false;
    if (!make_kv_tmap(&a.tmk, a.k_pool, p.kv_dtype, rows, D, S, &wk) ||
        !make_kv_tmap(&a.tmv, a.v_pool, p.kv_dtype, rows, D, S, &wv) || wk != wv)
      return cudaErrorNotSupported;
    a.whole_page = wk ? 1 : 0;
  }
  a.stages = stages;
  a.rows_per_stage = R;
  a.pages_per_stage = pps;
  a.stage_bytes = sb;
  a.row_bytes = rb;
  a.page_bytes = pb;
  a.ring_bytes = static_cast<uint32_t>(ring);
  a.keys_off = static_cast<uint32_t>(keys_off);
  a.sel_off = static_cast<uint32_t>(sel_off);
  a.att_off = static_cast<uint32_t>(att_off);

  auto kern = p.selector == SPG_SEL_QUEST ? k_fused<T, TQ, D, G, 0> : k_fused<T, TQ, D, G, 1>;
  cudaError_t e = ensure_smem(kern, smem);
  if (e != cudaSuccess) return e;
  // cluster size: 8 CTAs per unit when the GPU can hold them all at once,
  // else 4 or 2, so that the grid stays within about one wave
  const int units = p.batch * p.num_kv_heads;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  // the leader's copy of the page-table row, when it costs no occupancy (and
  // rows are 16-byte aligned for the bulk copy)
  a.pt_off = 0;
  if (p.max_pages_per_seq % 4 == 0) {
    const size_t pt_off = (smem - 1024 + 127) & ~static_cast<size_t>(127);
    const size_t smem_pt = 1024 + pt_off + sizeof(int) * p.max_pages_per_seq;
    int per_sm_pt = 0;
    if (smem_pt <= 227u * 1024u && ensure_smem(kern, smem_pt) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_pt, kern, threads, smem_pt) == cudaSuccess &&
        per_sm_pt >= per_sm) {
      a.pt_off = static_cast<uint32_t>(pt_off);
      smem = smem_pt;
    }
  }
  const int slots = device_sm_count() * per_sm;
  int C = kMaxCluster;
  while (C > 2 && units * C > slots) C /= 2;
  a.cluster = C;
  // sketch scan stages sized so that each consumer warp gets about one
  // stage of the CTA's chunk of blocks (the stage buffers stay as planned)
  if (p.selector == SPG_SEL_SKETCH_INT4) {
    const int cpc_max = (p.max_pages_per_seq + C - 1) / C;
    // (at most 32: a warp scores one block per lane)
    a.rows_per_stage = std::min(std::min(R, 32), std::max(4, (cpc_max + kConsumerWarps - 1) / kConsumerWarps));
  }
  // the sketch append gives each aux-warp lane one token of the block
  if (a.append && p.selector == SPG_SEL_SKETCH_INT4 && S > C * 32)
    return cudaErrorNotSupported;  // the caller falls back to the separate append
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(C, units);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // Load-balancing cluster placement: with the next step's CTAs launched
  // early (programmatic serialisation) the default placement can leave a
  // GPC's free slots too scattered for a whole cluster, and that cluster then
  // runs after the others, a full step late.
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  attr[2].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
  attr[2].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicyLoadBalancing;
  cfg.attrs = attr;
  cfg.numAttrs = 3;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, typename TQ>
cudaError_t fused_dispatch(const spg_params& p, const FusedArgs& a, cudaStream_t st) {
  const int G = p.num_q_heads / p.num_kv_heads;
#define SPG_FU(D_, G_) \
  if (p.head_dim == D_ && G == G_) return fused_typed<T, TQ, D_, G_>(p, a, st);
  SPG_FU(128, 1) SPG_FU(128, 2) SPG_FU(128, 4) SPG_FU(128, 8)
  SPG_FU(64, 1) SPG_FU(64, 2) SPG_FU(64, 4) SPG_FU(64, 8)
#undef SPG_FU
  return cudaErrorNotSupported;
}

}  // namespace

bool fused_supported(const spg_params& p, int append) {
  if (p.selector != SPG_SEL_QUEST && p.selector != SPG_SEL_SKETCH_INT4) return false;
  if (p.max_pages_per_seq > kFusedMaxPages) return false;
  if (p.selector == SPG_SEL_SKETCH_INT4 && p.page_size > 128) return false;
  if (append && p.n_recent_pages < 1) return false;  // the appended token's page must be forced
  if (append && p.selector == SPG_SEL_SKETCH_INT4 && p.sketch_dim != 16) return false;
  return true;
}

cudaError_t launch_fused(const spg_params& p, const void* q, const void* k_pool,
                         const void* v_pool, const void* k_scale, const void* v_scale,
                         const int32_t* page_table, const int32_t* seq_lens, void* minmax,
                         const uint8_t* sketch, const float* sketch_scale, const float* proj,
                         int32_t* sel, int32_t* sel_cnt, float* out, float* lse, int append,
                         const Workspace& ws, cudaStream_t stream) {
  FusedArgs a{};
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.k_scale = static_cast<const __half*>(k_scale);
  a.v_scale = static_cast<const __half*>(v_scale);
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.minmax = minmax;
  a.sketch = sketch;
  a.sketch_scale = sketch_scale;
  // with append, the caller (sparse_decode_step) owns writable sketch arrays
  a.sketch_w = append ? const_cast<uint8_t*>(sketch) : nullptr;
  a.sketch_scale_w = append ? const_cast<float*>(sketch_scale) : nullptr;
  a.proj = proj;
  a.sel = sel;
  a.sel_cnt = sel_cnt;
  a.out = out;
  a.lse = lse;
  a.err = ws.err;
  a.Hkv = p.num_kv_heads;
  a.S = p.page_size;
  a.MP = p.max_pages_per_seq;
  a.n_phys = p.num_phys_pages;
  a.n_sink = p.n_sink_pages;
  a.n_recent = p.n_recent_pages;
  a.n_sel = n_sel_pages(p);
  a.append = append;
  const float scale = p.softmax_scale > 0.f ? p.softmax_scale
                                            : 1.0f / sqrtf(static_cast<float>(p.head_dim));
  a.scale_log2 = scale * kLog2e;
  a.inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(p.head_dim));
  a.top_p = p.top_p;
  a.min_pages = p.min_pages;
  a.tau = p.selector == SPG_SEL_SKETCH_INT4 ? 1.0f : scale;
  switch (p.kv_dtype) {
    case SPG_F16:
      return fused_dispatch<__half, __half>(p, a, stream);
    case SPG_BF16:
      return fused_dispatch<__nv_bfloat16, __nv_bfloat16>(p, a, stream);
    default:
      if (p.q_dtype == SPG_F16) return fused_dispatch<int8_t, __half>(p, a, stream);
      return fused_dispatch<int8_t, __nv_bfloat16>(p, a, stream);
  }
}

}  // namespace spg
