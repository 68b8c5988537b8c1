// MLA prefill attention for one plan chunk, bf16, on pairs of SMs
// ("flare_mla_prefill_dispatch": q [tokens, H, 192], ragged k (nope) and v
// [rows, H, 128], k_rope [rows, 64] shared by all heads, causal mask offset by
// each sequence's cache length, log-sum-exp merge of per-chunk results).
//
// Same arithmetic and epilogue as attn_kernel; what changes is who loads what.
// A cluster of two CTAs (one per SM of a pair) takes a work item of two
// adjacent 128-row query tiles (2t, 2t+1) of one sequence and head: CTA r
// owns query tile 2t + r.  Both tiles visit the same key tiles, so every
// tcgen05.mma is a two-SM MMA (cta_group::2, M = 256): each CTA keeps its own
// Q rows, S/P and O in its TMEM, and holds HALF of every K tile (keys
// [64r, 64r + 64) of the tile, the N half of S = Q K^T) and half of every V
// tile (value columns [64r, 64r + 64), the N half of O += P V).  Each SM thus
// streams half of the K/V bytes per unit of tensor work, which is what bounds
// the one-SM kernel (the L2 -> SM stream), and the halved stages leave room
// for 4-deep rings.
//
//   warp 0      TMA: own Q tile (3 x 16 KB) into shared memory, own half of
//               each K tile (nope 2 x 8 KB + rope 8 KB), 4-stage ring.
//   warp 6      TMA: own half of each V tile (16 KB), 4-stage ring.
//   warp 1      both CTAs: TMEM allocation (512 columns, pair form).
//               CTA 0: one elected lane issues every MMA of the pair and
//               commits to the barriers of both CTAs.
//               CTA 1: one elected lane relays the completion of its K/V
//               halves to CTA 0's ring barriers, in the order the MMAs use them.
//   warps 2..5  softmax and epilogue of the CTA's own 128 query rows, exactly
//               as in attn_kernel; their "P ready", "Q staged" and "O read"
//               signals go to CTA 0's barriers.
//
// Work items whose tiles differ in key count run the larger count on both
// CTAs; the extra tile is fully masked for the shorter one (P = 0).
//
// TMEM columns (each CTA): S/P 0..127 and 128..255, O 256..383, Q 384..479.
#include <algorithm>
#include <mutex>

#include "attn_common.cuh"

namespace mla {
namespace {

constexpr int PBLK = 128 * 128;                 // 128 rows x 128 bytes (swizzled block)
constexpr int HBLK = 64 * 128;                  // 64 rows x 128 bytes
constexpr int PQ_BYTES = 3 * PBLK;              // own Q tile, 192 bf16 columns
constexpr int PK_BYTES = 3 * HBLK;              // half K tile: 64 keys x (128 nope + 64 rope)
constexpr int PV_BYTES = PBLK;                  // half V tile: 128 keys x 64 value columns
constexpr int PNK = 4, PNV = 4;
constexpr int P_SMEM_Q = 0;
constexpr int P_SMEM_K = P_SMEM_Q + PQ_BYTES;
constexpr int P_SMEM_V = P_SMEM_K + PNK * PK_BYTES;
constexpr int P_SMEM_BAR = P_SMEM_V + PNV * PV_BYTES;   // 212992
constexpr int P_SMEM_UNITS = P_SMEM_BAR + 256;                // compaction counts, then the unit list
constexpr int P_SMEM_TOTAL = P_SMEM_UNITS + 32 + 4 * 4096 + 1024;   // the largest launch
constexpr int P_THREADS = 224;
constexpr uint32_t P_TMEM_COLS = 512;
constexpr uint32_t P_TM_S = 0, P_TM_O = 256, P_TM_Q = 384;
constexpr uint32_t IDESC_QK2 = idesc_bf16(256, 128, false, false);
constexpr uint32_t IDESC_PV2 = idesc_bf16(256, 128, false, true);
constexpr uint16_t kBoth = 3;

struct PairSmem {
  uint64_t q_full, q_empty;   // own Q in shared memory
  uint64_t q_ready;           // CTA 0: both CTAs' Q in TMEM (8 warps)
  uint64_t k_full[PNK], k_empty[PNK];
  uint64_t v_full[PNV], v_empty[PNV];
  uint64_t s_full[2];
  uint64_t p_full[2];         // CTA 0: both CTAs' P in TMEM (8 warps)
  uint64_t o_done[2];         // o_done[t & 1] completes when P*V of tile t does
  uint64_t o_free;            // CTA 0: both CTAs read O (8 warps)
  uint64_t drain;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(PairSmem) <= 256, "barrier block");

// Work item of a pair: two adjacent query tiles of one sequence and head.
struct PairItem {
  Item own;    // this CTA's query tile
  int n_kv;    // key tiles both CTAs visit
};

// The chunk's work units (sequence b, query-tile pair tp) with work, in the
// order the items visit them (heaviest pairs first), compacted in shared
// memory by every CTA before the roles start.  Items are then (head group,
// unit, head) over that list, so the static stride of the clusters walks
// consecutive work and the clusters in flight stay within one head group and
// share its K/V in L2.  (Striding over all units instead lets the clusters
// drift into different head groups wherever most units of a chunk are empty,
// and K/V then comes from DRAM about twice.)  More than kMaxUnits units: the
// kernels walk all units and skip the empty ones.
constexpr int kMaxUnits = 4096;

// The 64 k_rope rows of a half tile from the paged cache, 16 bytes per
// cp.async: lane l holds cache rows ra (key l) and rb (key l + 32); each warp
// instruction copies 32 / CH whole rows (CH = 16-byte chunks per row), chunk
// l % CH of row RPI * i + l / CH, into the swizzled layout a tensor-map load
// would give (SW128 for 128-byte rows, SW64 for 64-byte rows; the tile base
// is aligned to the swizzle period).  Commits one cp.async group.
template <int ROW_BYTES>
__device__ __forceinline__ void rope_rows_cp_async(uint32_t dst, const uint8_t* rope_col0, int cache_row_bytes,
                                                   int ra, int rb) {
  constexpr int CH = ROW_BYTES / 16;
  constexpr int RPI = 32 / CH;
  constexpr int ITERS = 64 / RPI;
  const int lane = threadIdx.x & 31;
  const int c = lane % CH;
  const uint8_t* src = rope_col0 + c * 16;
#pragma unroll
  for (int i = 0; i < ITERS; ++i) {
    const int r = RPI * i + lane / CH;
    const int row = __shfl_sync(0xffffffffu, i < ITERS / 2 ? ra : rb, r & 31);
    const int sw = ROW_BYTES == 128 ? (r & 7) : ((r >> 1) & 3);
    cp_async16(dst + r * ROW_BYTES + ((c ^ sw) << 4), src + static_cast<size_t>(row) * cache_row_bytes);
  }
  cp_async_commit();
}

// The k_rope copies of a stage have landed (all but the newest PENDING
// cp.async groups of the warp): fence them into the async proxy the MMAs
// read through, then count them on the stage's barrier `bar`.
template <int PENDING>
__device__ __forceinline__ void rope_rows_landed(uint32_t bar) {
  cp_async_wait<PENDING>();
  fence_async_smem();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

struct WorkList {
  const uint32_t* units;   // shared memory
  int n;                   // units with work, or -1: walk all units
};

__device__ __forceinline__ bool load_pair(const Params& p, int idx, uint32_t rank, PairItem& it,
                                          const WorkList& wl) {
  const int n_tp = (p.n_qtiles + 1) >> 1;   // tile pairs per sequence
  const int n_units = wl.n >= 0 ? wl.n : n_tp * p.B;
  const int per_group = p.head_group * n_units;
  const int grp = idx / per_group;
  const int r = idx - grp * per_group;
  const int hg = min(p.head_group, p.H - grp * p.head_group);
  const int ui = r / hg;
  const int h = grp * p.head_group + (r - ui * hg);
  const int unit = wl.n >= 0 ? static_cast<int>(wl.units[ui]) : ui;
  const int tp = n_tp - 1 - unit / p.B;   // heaviest pairs first
  const int b = unit % p.B;
  Item other;
  tile_item(p, b, h, 2 * tp + static_cast<int>(rank), it.own);
  tile_item(p, b, h, 2 * tp + 1 - static_cast<int>(rank), other);
  it.n_kv = max(it.own.n_kv, other.n_kv);
  return it.n_kv > 0;
}

__device__ __forceinline__ bool next_pair(const Params& p, int& idx, int stride, int total, uint32_t rank,
                                          PairItem& it, const WorkList& wl) {
  for (; idx < total; idx += stride)
    if (load_pair(p, idx, rank, it, wl)) return true;
  return false;
}

// Every thread of the CTA: compact the units with work into `list`; returns
// their count (the same in every thread), or -1 past kMaxUnits.
__device__ int compact_units(const Params& p, uint32_t* list, int* warp_cnt) {
  const int n_tp = (p.n_qtiles + 1) >> 1;
  const int n_units = n_tp * p.B;
  if (n_units > kMaxUnits) return -1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nwarps = static_cast<int>(blockDim.x) >> 5;
  int base = 0;
  for (int u0 = 0; u0 < n_units; u0 += static_cast<int>(blockDim.x)) {
    const int u = u0 + tid;
    bool has = false;
    if (u < n_units) {
      const int tp = n_tp - 1 - u / p.B, b = u % p.B;
      Item a, c;
      tile_item(p, b, 0, 2 * tp, a);
      tile_item(p, b, 0, 2 * tp + 1, c);
      has = max(a.n_kv, c.n_kv) > 0;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, has);
    if (lane == 0) warp_cnt[warp] = __popc(m);
    __syncthreads();
    int off = base, tot = 0;
    for (int w = 0; w < nwarps; ++w) {
      if (w < warp) off += warp_cnt[w];
      tot += warp_cnt[w];
    }
    if (has) list[off + __popc(m & ((1u << lane) - 1u))] = static_cast<uint32_t>(u);
    base += tot;
    __syncthreads();   // warp_cnt is rewritten by the next round
  }
  return base;
}

// PAGED: k_rope from the paged cache through the chunk's cache-row table
// (an instantiation of its own, so that the buffered one carries no trace of it).
template <bool PAGED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap kn_map,
                     const __grid_constant__ CUtensorMap kr_map, const __grid_constant__ CUtensorMap v_map,
                     const Params p, int total_items, const PagedRope pr) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairSmem* sh = reinterpret_cast<PairSmem*>(smem + P_SMEM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair_id = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;

  pdl_enter();
  // Both CTAs of a pair see the same chunk length, so they return together.
  if (p.bl[p.chunk] <= 0) return;

  if (threadIdx.x == 0) {
    const uint32_t lead = rank == 0 ? 1u : 0u;
    mbar_init(smem_u32(&sh->q_full), 1);
    mbar_init(smem_u32(&sh->q_empty), 4);
    mbar_init(smem_u32(&sh->q_ready), 8);
    for (int i = 0; i < PNK; ++i) {
      // own bytes (+ the paged k_rope rows) + in CTA 0 the relay
      mbar_init(smem_u32(&sh->k_full[i]), 1 + lead + (PAGED ? 1u : 0u));
      mbar_init(smem_u32(&sh->k_empty[i]), 1);
    }
    for (int i = 0; i < PNV; ++i) {
      mbar_init(smem_u32(&sh->v_full[i]), 1 + lead);
      mbar_init(smem_u32(&sh->v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh->s_full[i]), 1);
      mbar_init(smem_u32(&sh->p_full[i]), 8);
      mbar_init(smem_u32(&sh->o_done[i]), 1);
    }
    mbar_init(smem_u32(&sh->o_free), 8);
    mbar_init(smem_u32(&sh->drain), 1);
    // A pipeline timeout recorded by an earlier kernel on this status word:
    // do no work (the pair agrees through cluster_any below).
    sh->abort = timed_out_before(p.status) ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&sh->tmem), P_TMEM_COLS);
    tmem_relinquish_pair();
  }
  // Compaction counts (8 ints), then the list, sized by the launch.
  const WorkList wl{reinterpret_cast<const uint32_t*>(smem + P_SMEM_UNITS + 32),
                    compact_units(p, reinterpret_cast<uint32_t*>(smem + P_SMEM_UNITS + 32),
                                  reinterpret_cast<int*>(smem + P_SMEM_UNITS))};
  tc_fence_before();
  cluster_sync();   // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const int total = cluster_any(&sh->abort) ? 0 : (wl.n >= 0 ? wl.n * p.H : total_items);
  const uint32_t tmem = sh->tmem;
  volatile int* abort_flag = &sh->abort;
  int32_t* status = p.status;

  if (warp == 0) {
    // ------------------------------------------------------------ Q and K producer
    if (elect_one()) {
      prefetch_tmap(&q_map);
      prefetch_tmap(&kn_map);
      prefetch_tmap(&kr_map);
    }
    __syncwarp();
    uint32_t g = 0, it_n = 0;
    int q_last = -1, k_last[PNK] = {-1, -1, -1, -1};
    int k_pend = -1;   // stage whose paged k_rope rows are in flight
    bool ok = true;
    PairItem it;
    for (int idx = pair_id; ok && next_pair(p, idx, n_pairs, total, rank, it, wl); idx += n_pairs) {
      if (it_n > 0 && !(ok = mbar_wait_warp(smem_u32(&sh->q_empty), (it_n - 1) & 1, status, abort_flag))) break;
      if (elect_one()) {
        const uint32_t qf = smem_u32(&sh->q_full);
        mbar_expect_tx(qf, PQ_BYTES);
        for (int blk = 0; blk < 3; ++blk)
          tma_load_2d(smem_u32(smem + P_SMEM_Q + blk * PBLK), &q_map, qf, it.own.h * 192 + blk * 64,
                      it.own.q_row0);
      }
      __syncwarp();
      q_last = int(it_n & 1);
      // Paged k_rope: table entries of the half tile's 64 keys (two a lane),
      // loaded a stage ahead of their use.
      int ra = 0, rb = 0;
      if constexpr (PAGED) {
        ra = cache_row_entry(pr, it.own, static_cast<int>(rank) * 64 + lane);
        rb = cache_row_entry(pr, it.own, static_cast<int>(rank) * 64 + 32 + lane);
      }
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t gj = g + j;
        const int row = it.own.kv_row0 + j * BN + static_cast<int>(rank) * 64;
        const int ks = gj % PNK;
        if (gj >= PNK &&
            !(ok = mbar_wait_cluster_warp(smem_u32(&sh->k_empty[ks]), ((gj / PNK) & 1) ^ 1, status, abort_flag)))
          break;
        const uint32_t kf = smem_u32(&sh->k_full[ks]);
        const uint32_t kdst = smem_u32(smem + P_SMEM_K + ks * PK_BYTES);
        if (elect_one()) {
          mbar_expect_tx(kf, PAGED ? 2 * HBLK : PK_BYTES);
          tma_load_2d(kdst, &kn_map, kf, it.own.h * 128, row);
          tma_load_2d(kdst + HBLK, &kn_map, kf, it.own.h * 128 + 64, row);
          if constexpr (!PAGED) tma_load_2d(kdst + 2 * HBLK, &kr_map, kf, 0, row);
        }
        __syncwarp();
        if constexpr (PAGED) {
          // k_rope rows by cp.async (one-row TMA gathers cost far more per
          // byte); the previous stage's rows are counted once they land.
          rope_rows_cp_async<128>(kdst + 2 * HBLK, pr.kv_cache + 1024, pr.cache_row_bytes, checked_cache_row(p, pr, ra),
                                     checked_cache_row(p, pr, rb));
          if (j + 1 < it.n_kv) {
            const int k1 = (j + 1) * BN + static_cast<int>(rank) * 64;
            ra = cache_row_entry(pr, it.own, k1 + lane);
            rb = cache_row_entry(pr, it.own, k1 + 32 + lane);
          }
          if (k_pend >= 0) rope_rows_landed<1>(smem_u32(&sh->k_full[k_pend]));
          k_pend = ks;
        }
        k_last[ks] = int((gj / PNK) & 1);
      }
      // The item's last k_rope rows, before any other wait.
      if (k_pend >= 0) rope_rows_landed<0>(smem_u32(&sh->k_full[k_pend]));
      k_pend = -1;
      g += it.n_kv;
      ++it_n;
    }
    if (k_pend >= 0) rope_rows_landed<0>(smem_u32(&sh->k_full[k_pend]));
    // Drain: every issued load lands before the CTA leaves.  (In CTA 0 the
    // K barriers also count the relay's arrival, so wait on the bytes only
    // through the phases this warp started: a bounded wait either way.)
    volatile int never = 0;
    if (q_last >= 0) mbar_wait_warp(smem_u32(&sh->q_full), uint32_t(q_last), status, &never);
    for (int s = 0; s < PNK; ++s)
      if (k_last[s] >= 0) mbar_wait_cluster_warp(smem_u32(&sh->k_full[s]), uint32_t(k_last[s]), status, &never);
    // ... and every stage release the pair MMAs multicast to this CTA has
    // arrived: an asynchronous arrival must not reach a CTA that has left.
    for (int s = 0; s < PNK; ++s)
      if (k_last[s] >= 0) mbar_wait_cluster_warp(smem_u32(&sh->k_empty[s]), uint32_t(k_last[s]), status, abort_flag);
  } else if (warp == 6) {
    // ------------------------------------------------------------ V producer
    if (elect_one()) prefetch_tmap(&v_map);
    __syncwarp();
    uint32_t g = 0;
    int v_last[PNV] = {-1, -1, -1, -1};
    bool ok = true;
    PairItem it;
    for (int idx = pair_id; ok && next_pair(p, idx, n_pairs, total, rank, it, wl); idx += n_pairs) {
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t gj = g + j;
        const int row = it.own.kv_row0 + j * BN;
        const int vs = gj % PNV;
        if (gj >= PNV &&
            !(ok = mbar_wait_cluster_warp(smem_u32(&sh->v_empty[vs]), ((gj / PNV) & 1) ^ 1, status, abort_flag)))
          break;
        if (elect_one()) {
          const uint32_t vf = smem_u32(&sh->v_full[vs]);
          mbar_expect_tx(vf, PV_BYTES);
          tma_load_2d(smem_u32(smem + P_SMEM_V + vs * PV_BYTES), &v_map, vf,
                      it.own.h * 128 + static_cast<int>(rank) * 64, row);
        }
        __syncwarp();
        v_last[vs] = int((gj / PNV) & 1);
      }
      g += it.n_kv;
    }
    volatile int never = 0;
    for (int s = 0; s < PNV; ++s)
      if (v_last[s] >= 0) mbar_wait_cluster_warp(smem_u32(&sh->v_full[s]), uint32_t(v_last[s]), status, &never);
    for (int s = 0; s < PNV; ++s)
      if (v_last[s] >= 0) mbar_wait_cluster_warp(smem_u32(&sh->v_empty[s]), uint32_t(v_last[s]), status, abort_flag);
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------------------------------------------------- pair MMA issuer
      // One elected lane runs the whole loop (no reconvergence while MMAs are
      // in flight); every commit goes to the barrier in both CTAs.
      if (elect_one()) {
        uint32_t g = 0, it_n = 0;
        const uint32_t q_t = tmem + P_TM_Q;
        const uint32_t o_t = tmem + P_TM_O;
        PairItem it;
        for (int idx = pair_id; next_pair(p, idx, n_pairs, total, rank, it, wl); idx += n_pairs) {
          if (!mbar_wait_cluster(smem_u32(&sh->q_ready), it_n & 1, status, abort_flag)) break;
          const int n = it.n_kv;
          auto issue_s = [&](int j) -> bool {
            const uint32_t gj = g + j;
            const int ks = gj % PNK;
            if (!mbar_wait_cluster(smem_u32(&sh->k_full[ks]), (gj / PNK) & 1, status, abort_flag)) return false;
            tc_fence_after();
            const uint32_t k_s = smem_u32(smem + P_SMEM_K + ks * PK_BYTES);
            const uint32_t d = tmem + P_TM_S + (gj & 1) * 128;
#pragma unroll
            for (int kk = 0; kk < 12; ++kk) {
              const uint32_t off = (kk >> 2) * HBLK + (kk & 3) * 32;
              mma_f16_ts_pair(d, q_t + kk * 8, sdesc(k_s + off, 16, 1024), IDESC_QK2, kk > 0);
            }
            tc_commit_pair(smem_u32(&sh->s_full[gj & 1]), kBoth);
            tc_commit_pair(smem_u32(&sh->k_empty[ks]), kBoth);
            return true;
          };
          auto issue_pv = [&](int j) -> bool {
            const uint32_t gp = g + j;
            const int vs = gp % PNV;
            // V and the free O first: they are ready long before P as a rule,
            // and checking them after P would add their barrier round trips to
            // the hand-off from the softmax to P*V.
            if (!mbar_wait_cluster(smem_u32(&sh->v_full[vs]), (gp / PNV) & 1, status, abort_flag)) return false;
            if (j == 0 && it_n >= 1 &&
                !mbar_wait_cluster(smem_u32(&sh->o_free), (it_n - 1) & 1, status, abort_flag))
              return false;
            if (!mbar_wait_cluster(smem_u32(&sh->p_full[gp & 1]), (gp >> 1) & 1, status, abort_flag)) return false;
            tc_fence_after();
            const uint32_t v_s = smem_u32(smem + P_SMEM_V + vs * PV_BYTES);
            const uint32_t pa = tmem + P_TM_S + (gp & 1) * 128;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_f16_ts_pair(o_t, pa + kk * 8, sdesc(v_s + kk * 2048, PBLK, 1024), IDESC_PV2, (j > 0 || kk > 0));
            tc_commit_pair(smem_u32(&sh->o_done[gp & 1]), kBoth);
            tc_commit_pair(smem_u32(&sh->v_empty[vs]), kBoth);
            return true;
          };
          bool ok = issue_s(0);
          if (ok && n > 1) ok = issue_s(1);
          for (int j = 0; j < n && ok; ++j) {
            ok = issue_pv(j);
            if (ok && j + 2 < n) ok = issue_s(j + 2);
          }
          if (!ok) break;
          g += n;
          ++it_n;
        }
        tc_commit_pair(smem_u32(&sh->drain), 1);
        volatile int never = 0;
        mbar_wait(smem_u32(&sh->drain), 0, status, &never);
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------------- relay (CTA 1)
      // Forward "my half of K_j / V_j has landed" to CTA 0's ring barriers in
      // the order CTA 0's MMAs consume them: K_0, K_1, then V_j, K_{j+2}.
      if (elect_one()) {
        const uint32_t k_full0 = cluster_addr(smem_u32(&sh->k_full[0]), 0);
        const uint32_t v_full0 = cluster_addr(smem_u32(&sh->v_full[0]), 0);
        uint32_t g = 0;
        PairItem it;
        auto relay_k = [&](uint32_t gj) -> bool {
          const int ks = gj % PNK;
          if (!mbar_wait(smem_u32(&sh->k_full[ks]), (gj / PNK) & 1, status, abort_flag)) return false;
          mbar_arrive_cluster(k_full0 + ks * 8);
          return true;
        };
        auto relay_v = [&](uint32_t gj) -> bool {
          const int vs = gj % PNV;
          if (!mbar_wait(smem_u32(&sh->v_full[vs]), (gj / PNV) & 1, status, abort_flag)) return false;
          mbar_arrive_cluster(v_full0 + vs * 8);
          return true;
        };
        for (int idx = pair_id; next_pair(p, idx, n_pairs, total, rank, it, wl); idx += n_pairs) {
          const int n = it.n_kv;
          bool ok = relay_k(g);
          if (ok && n > 1) ok = relay_k(g + 1);
          for (int j = 0; j < n && ok; ++j) {
            ok = relay_v(g + j);
            if (ok && j + 2 < n) ok = relay_k(g + j + 2);
          }
          if (!ok) break;
          g += n;
        }
      }
      __syncwarp();
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ softmax + epilogue
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    const float sl2 = p.scale_log2;
    const float2 sl2v = make_float2(sl2, sl2);
    const uint32_t q_ready0 = cluster_addr(smem_u32(&sh->q_ready), 0);
    const uint32_t p_full0 = cluster_addr(smem_u32(&sh->p_full[0]), 0);
    const uint32_t o_free0 = cluster_addr(smem_u32(&sh->o_free), 0);
    uint32_t g = 0, it_n = 0;
    bool ok = true;

    auto stage_q = [&](uint32_t n) -> bool {
      if (!mbar_wait_warp(smem_u32(&sh->q_full), n & 1, status, abort_flag)) return false;
      uint32_t v[96];
      const uint8_t* qs = smem + P_SMEM_Q + row * 128;
#pragma unroll
      for (int j = 0; j < 24; ++j) {
        const uint4 x = *reinterpret_cast<const uint4*>(qs + (j >> 3) * PBLK + (((j & 7) ^ (row & 7)) << 4));
        v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
      }
      tmem_st32(tmem + lane_off + P_TM_Q, v);
      tmem_st32(tmem + lane_off + P_TM_Q + 32, v + 32);
      tmem_st32(tmem + lane_off + P_TM_Q + 64, v + 64);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh->q_empty));
        mbar_arrive_cluster(q_ready0);
      }
      return true;
    };

    int idx = pair_id;
    PairItem it;
    bool have = next_pair(p, idx, n_pairs, total, rank, it, wl);
    if (have) ok = stage_q(0);
    while (have && ok) {
      const Item& own = it.own;
      const long long qpos = static_cast<long long>(own.cb) + own.i0 + row;
      const long long lim_all = min(static_cast<long long>(own.n_cb), qpos - own.co + 1);
      float m_run = kNegInf, l_run = 0.f;
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t gj = g + j;
        const uint32_t sb = gj & 1;
        if (!(ok = mbar_wait_cluster_warp(smem_u32(&sh->s_full[sb]), (gj >> 1) & 1, status, abort_flag))) break;
        tc_fence_after();
        float x[BN];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tmem + lane_off + P_TM_S + sb * 128 + c * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(reinterpret_cast<uint32_t*>(x) + c * 32));
        tmem_ld_wait();
        const long long lim = lim_all - static_cast<long long>(j) * BN;
        if (lim < BN) {
#pragma unroll
          for (int k = 0; k < BN; ++k) x[k] = k < lim ? x[k] : kNegInf;
        }
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmax3(x[i], x[8 + i], x[16 + i]);
#pragma unroll
        for (int k = 24; k + 16 <= BN; k += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], x[k + i], x[k + 8 + i]);
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], x[BN - 8 + i]);
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7]));
        const float m_new = fmaxf(m_run, mx * sl2);
        const bool need = m_new > m_run + kRescaleThreshold;
        const float f = need ? ex2(m_run - m_new) : 1.0f;
        if (need) m_run = m_new;
        const float msub = m_run == kNegInf ? 0.f : m_run;
        const float2 negm = make_float2(-msub, -msub);
        uint32_t pk[BN / 2];
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int k = 0; k < BN / 2; ++k) {
          const float2 t = __ffma2_rn(make_float2(x[2 * k], x[2 * k + 1]), sl2v, negm);
          const float2 e = make_float2(ex2(t.x), ex2(t.y));
          acc[k & 3] = __fadd2_rn(acc[k & 3], e);
          pk[k] = pack_bf16(e.x, e.y);
        }
        const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
        const float2 a = __fadd2_rn(a01, a23);
        l_run = l_run * f + (a.x + a.y);
        if (j == it.n_kv - 1 && own.n_cb - j * BN < BN) {
          // Keys past the sequence in the last tile: zero this CTA's half of
          // those V rows (stale or non-finite) before P*V reads them.
          const int vs = gj % PNV;
          if (!(ok = mbar_wait_cluster_warp(smem_u32(&sh->v_full[vs]), (gj / PNV) & 1, status, abort_flag))) break;
          if (j * BN + row >= own.n_cb) {
            uint8_t* vrow = smem + P_SMEM_V + vs * PV_BYTES + row * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) reinterpret_cast<uint4*>(vrow)[c] = make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
        }
        tmem_st64(tmem + lane_off + P_TM_S + sb * 128, pk);
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // Rescale O only when the row maximum grew by more than 2^8, once P*V
          // of the previous tile has completed.
          if (!(ok = mbar_wait_cluster_warp(smem_u32(&sh->o_done[(gj - 1) & 1]), ((gj - 1) >> 1) & 1, status,
                                            abort_flag)))
            break;
          {
            tc_fence_after();
            uint32_t r[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t ta = tmem + lane_off + P_TM_O + c * 32;
              tmem_ld32(ta, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
              tmem_st32(ta, r);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(p_full0 + sb * 8);
      }
      if (!ok) break;
      g += it.n_kv;
      int nidx = idx + n_pairs;
      PairItem nx;
      const bool have_next = next_pair(p, nidx, n_pairs, total, rank, nx, wl);
      if (have_next && !(ok = stage_q(it_n + 1))) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = mbar_wait_cluster_warp(smem_u32(&sh->o_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, status,
                                        abort_flag)))
        break;
      tc_fence_after();
      float o[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld32(tmem + lane_off + P_TM_O + c * 32,
                  *reinterpret_cast<uint32_t(*)[32]>(reinterpret_cast<uint32_t*>(o) + c * 32));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(o_free0);
      const Item cur = it.own;
      it = nx;
      idx = nidx;
      have = have_next;
      ++it_n;
      store_row(p, cur, row, qpos, m_run, l_run, o);
    }
    // The completion of the P*V before the last (the other o_done barrier)
    // has arrived too: no asynchronous arrival may reach a CTA that has left.
    if (ok && g >= 2)
      mbar_wait_cluster_warp(smem_u32(&sh->o_done[(g - 2) & 1]), ((g - 2) >> 1) & 1, status, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // neither CTA frees TMEM or leaves while the pair still uses it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, P_TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// e4m3 inputs.  The same pair schedule; Q and K are e4m3 and S = Q K^T runs as
// kind::f8f6f4 pair MMAs with both operands in shared memory (Q double
// buffered, since the MMAs read it there: nope part 128-byte swizzled, rope
// part 64-byte swizzled); V arrives as f16 holding the e4m3-rounded values
// (written so by the up-projection), and P is f16, so P V is a kind::f16 pair
// MMA with no widening in this kernel.
constexpr int EQN_BYTES = 128 * 128;            // Q nope: 128 rows x 128 B
constexpr int EQ_BYTES = EQN_BYTES + 128 * 64;  // + rope: 128 rows x 64 B
constexpr int EKN_BYTES = 64 * 128;             // K nope half: 64 keys x 128 B
constexpr int EK_BYTES = EKN_BYTES + 64 * 64;   // + rope: 64 keys x 64 B
constexpr int E_SMEM_Q = 0;                                  // 2 slots
constexpr int E_SMEM_K = E_SMEM_Q + 2 * EQ_BYTES;
constexpr int E_SMEM_V = E_SMEM_K + PNK * EK_BYTES;          // f16 halves, as in the bf16 kernel
constexpr int E_SMEM_BAR = E_SMEM_V + PNV * PV_BYTES;        // 163840
constexpr int E_SMEM_UNITS = E_SMEM_BAR + 256;                // compaction counts, then the unit list
constexpr int E_SMEM_TOTAL = E_SMEM_UNITS + 32 + 4 * 4096 + 1024;   // the largest launch
constexpr uint32_t IDESC_QK8P = idesc_e4m3(256, 128, false, false);
constexpr uint32_t IDESC_PV16P = idesc_f16(256, 128, false, true);
static_assert(EQ_BYTES % 1024 == 0 && EK_BYTES % 1024 == 0 && E_SMEM_V % 1024 == 0, "swizzle alignment");

struct PairSmem8 {
  uint64_t q_full[2];         // own Q landed in slot n & 1
  uint64_t q_free[2];         // slot free: the item's last S MMA completed
  uint64_t q_ready;           // CTA 0: both CTAs' Q landed (8 warps)
  uint64_t k_full[PNK], k_empty[PNK];
  uint64_t v_full[PNV], v_empty[PNV];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t o_free;
  uint64_t drain;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(PairSmem8) <= 256, "barrier block");

template <bool PAGED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
    attn_pair_kernel_e4m3(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap qr_map,
                          const __grid_constant__ CUtensorMap kn_map, const __grid_constant__ CUtensorMap kr_map,
                          const __grid_constant__ CUtensorMap v_map, const Params p, int total_items,
                          const PagedRope pr) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairSmem8* sh = reinterpret_cast<PairSmem8*>(smem + E_SMEM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair_id = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;

  pdl_enter();
  // Both CTAs of a pair see the same chunk length, so they return together.
  if (p.bl[p.chunk] <= 0) return;

  if (threadIdx.x == 0) {
    const uint32_t lead = rank == 0 ? 1u : 0u;
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh->q_full[i]), 1);
      mbar_init(smem_u32(&sh->q_free[i]), 1);
    }
    mbar_init(smem_u32(&sh->q_ready), 8);
    for (int i = 0; i < PNK; ++i) {
      // own bytes (+ the paged k_rope rows) + in CTA 0 the relay
      mbar_init(smem_u32(&sh->k_full[i]), 1 + lead + (PAGED ? 1u : 0u));
      mbar_init(smem_u32(&sh->k_empty[i]), 1);
    }
    for (int i = 0; i < PNV; ++i) {
      mbar_init(smem_u32(&sh->v_full[i]), 1 + lead);
      mbar_init(smem_u32(&sh->v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh->s_full[i]), 1);
      mbar_init(smem_u32(&sh->p_full[i]), 8);
      mbar_init(smem_u32(&sh->o_done[i]), 1);
    }
    mbar_init(smem_u32(&sh->o_free), 8);
    mbar_init(smem_u32(&sh->drain), 1);
    // A pipeline timeout recorded by an earlier kernel on this status word:
    // do no work (the pair agrees through cluster_any below).
    sh->abort = timed_out_before(p.status) ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&sh->tmem), P_TMEM_COLS);
    tmem_relinquish_pair();
  }
  // Compaction counts (8 ints), then the list, sized by the launch.
  const WorkList wl{reinterpret_cast<const uint32_t*>(smem + E_SMEM_UNITS + 32),
                    compact_units(p, reinterpret_cast<uint32_t*>(smem + E_SMEM_UNITS + 32),
                                  reinterpret_cast<int*>(smem + E_SMEM_UNITS))};
  tc_fence_before();
  cluster_sync();   // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const int total = cluster_any(&sh->abort) ? 0 : (wl.n >= 0 ? wl.n * p.H : total_items);
  const uint32_t tmem = sh->tmem;
  volatile int* abort_flag = &sh->abort;
  int32_t* status = p.status;

  if (warp == 0) {
    // ------------------------------------------------------------ Q and K producer
    if (elect_one()) {
      prefetch_tmap(&q_map);
      prefetch_tmap(&qr_map);
      prefetch_tmap(&kn_map);
      prefetch_tmap(&kr_map);
    }
    __syncwarp();
    uint32_t g = 0, it_n = 0;
    int q_last[2] = {-1, -1}, k_last[PNK] = {-1, -1, -1, -1};
    int k_pend = -1;   // stage whose paged k_rope rows are in flight
    bool ok = true;
    PairItem it;
    for (int idx = pair_id; ok && next_pair(p, idx, n_pairs, total, rank, it, wl); idx += n_pairs) {
      // Q slot it_n & 1 is free once item it_n - 2's last S MMA completed
      // (the MMAs read Q from shared memory).
      const int qs = it_n & 1;
      if (it_n > 1 &&
          !(ok = mbar_wait_cluster_warp(smem_u32(&sh->q_free[qs]), ((it_n - 2) >> 1) & 1, status, abort_flag)))
        break;
      if (elect_one()) {
        const uint32_t qf = smem_u32(&sh->q_full[qs]);
        const uint32_t qd = smem_u32(smem + E_SMEM_Q + qs * EQ_BYTES);
        mbar_expect_tx(qf, EQ_BYTES);
        tma_load_2d(qd, &q_map, qf, it.own.h * 192, it.own.q_row0);              // nope: 128 B a row
        tma_load_2d(qd + EQN_BYTES, &qr_map, qf, it.own.h * 192 + 128, it.own.q_row0);   // rope: 64 B
      }
      __syncwarp();
      q_last[qs] = int((it_n >> 1) & 1);
      // Paged k_rope: table entries of the half tile's 64 keys (two a lane),
      // loaded a stage ahead of their use.
      int ra = 0, rb = 0;
      if constexpr (PAGED) {
        ra = cache_row_entry(pr, it.own, static_cast<int>(rank) * 64 + lane);
        rb = cache_row_entry(pr, it.own, static_cast<int>(rank) * 64 + 32 + lane);
      }
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t gj = g + j;
        const int row = it.own.kv_row0 + j * BN + static_cast<int>(rank) * 64;
        const int ks = gj % PNK;
        if (gj >= PNK &&
            !(ok = mbar_wait_cluster_warp(smem_u32(&sh->k_empty[ks]), ((gj / PNK) & 1) ^ 1, status, abort_flag)))
          break;
        const uint32_t kf = smem_u32(&sh->k_full[ks]);
        const uint32_t kdst = smem_u32(smem + E_SMEM_K + ks * EK_BYTES);
        if (elect_one()) {
          mbar_expect_tx(kf, PAGED ? EKN_BYTES : EK_BYTES);
          tma_load_2d(kdst, &kn_map, kf, it.own.h * 128, row);      // nope: 64 keys x 128 B
          if constexpr (!PAGED) tma_load_2d(kdst + EKN_BYTES, &kr_map, kf, 0, row);   // rope: 64 keys x 64 B
        }
        __syncwarp();
        if constexpr (PAGED) {   // as in the bf16 kernel
          rope_rows_cp_async<64>(kdst + EKN_BYTES, pr.kv_cache + 512, pr.cache_row_bytes, checked_cache_row(p, pr, ra),
                                     checked_cache_row(p, pr, rb));
          if (j + 1 < it.n_kv) {
            const int k1 = (j + 1) * BN + static_cast<int>(rank) * 64;
            ra = cache_row_entry(pr, it.own, k1 + lane);
            rb = cache_row_entry(pr, it.own, k1 + 32 + lane);
          }
          if (k_pend >= 0) rope_rows_landed<1>(smem_u32(&sh->k_full[k_pend]));
          k_pend = ks;
        }
        k_last[ks] = int((gj / PNK) & 1);
      }
      if (k_pend >= 0) rope_rows_landed<0>(smem_u32(&sh->k_full[k_pend]));
      k_pend = -1;
      g += it.n_kv;
      ++it_n;
    }
    if (k_pend >= 0) rope_rows_landed<0>(smem_u32(&sh->k_full[k_pend]));
    // Drain: every issued load lands before the CTA leaves.  (In CTA 0 the
    // K barriers also count the relay's arrival, so wait on the bytes only
    // through the phases this warp started: a bounded wait either way.)
    volatile int never = 0;
    for (int s = 0; s < 2; ++s)
      if (q_last[s] >= 0) mbar_wait_warp(smem_u32(&sh->q_full[s]), uint32_t(q_last[s]), status, &never);
    for (int s = 0; s < PNK; ++s)
      if (k_last[s] >= 0) mbar_wait_cluster_warp(smem_u32(&sh->k_full[s]), uint32_t(k_last[s]), status, &never);
    // ... and every slot and stage release the pair MMAs multicast to this CTA
    // has arrived: an asynchronous arrival must not reach a CTA that has left.
    for (int s = 0; s < 2; ++s)
      if (q_last[s] >= 0) mbar_wait_cluster_warp(smem_u32(&sh->q_free[s]), uint32_t(q_last[s]), status, abort_flag);
    for (int s = 0; s < PNK; ++s)
      if (k_last[s] >= 0) mbar_wait_cluster_warp(smem_u32(&sh->k_empty[s]), uint32_t(k_last[s]), status, abort_flag);
  } else if (warp == 6) {
    // ------------------------------------------------------------ V producer
    if (elect_one()) prefetch_tmap(&v_map);
    __syncwarp();
    uint32_t g = 0;
    int v_last[PNV] = {-1, -1, -1, -1};
    bool ok = true;
    PairItem it;
    for (int idx = pair_id; ok && next_pair(p, idx, n_pairs, total, rank, it, wl); idx += n_pairs) {
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t gj = g + j;
        const int row = it.own.kv_row0 + j * BN;
        const int vs = gj % PNV;
        if (gj >= PNV &&
            !(ok = mbar_wait_cluster_warp(smem_u32(&sh->v_empty[vs]), ((gj / PNV) & 1) ^ 1, status, abort_flag)))
          break;
        if (elect_one()) {
          const uint32_t vf = smem_u32(&sh->v_full[vs]);
          mbar_expect_tx(vf, PV_BYTES);
          tma_load_2d(smem_u32(smem + E_SMEM_V + vs * PV_BYTES), &v_map, vf,
                      it.own.h * 128 + static_cast<int>(rank) * 64, row);
        }
        __syncwarp();
        v_last[vs] = int((gj / PNV) & 1);
      }
      g += it.n_kv;
    }
    volatile int never = 0;
    for (int s = 0; s < PNV; ++s)
      if (v_last[s] >= 0) mbar_wait_cluster_warp(smem_u32(&sh->v_full[s]), uint32_t(v_last[s]), status, &never);
    for (int s = 0; s < PNV; ++s)
      if (v_last[s] >= 0) mbar_wait_cluster_warp(smem_u32(&sh->v_empty[s]), uint32_t(v_last[s]), status, abort_flag);
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------------------------------------------------- pair MMA issuer
      // One elected lane runs the whole loop (no reconvergence while MMAs are
      // in flight); every commit goes to the barrier in both CTAs.
      if (elect_one()) {
        uint32_t g = 0, it_n = 0;
        const uint32_t o_t = tmem + P_TM_O;
        PairItem it;
        for (int idx = pair_id; next_pair(p, idx, n_pairs, total, rank, it, wl); idx += n_pairs) {
          if (!mbar_wait_cluster(smem_u32(&sh->q_ready), it_n & 1, status, abort_flag)) break;
          const int n = it.n_kv;
          auto issue_s = [&](int j) -> bool {
            const uint32_t gj = g + j;
            const int ks = gj % PNK;
            if (!mbar_wait_cluster(smem_u32(&sh->k_full[ks]), (gj / PNK) & 1, status, abort_flag)) return false;
            tc_fence_after();
            const uint32_t k_s = smem_u32(smem + E_SMEM_K + ks * EK_BYTES);
            const uint32_t q_s = smem_u32(smem + E_SMEM_Q + (it_n & 1) * EQ_BYTES);
            const uint32_t d = tmem + P_TM_S + (gj & 1) * 128;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)   // nope: 128 B a row, 32 e4m3 per MMA
              mma_f8_ss_pair(d, sdesc(q_s + kk * 32, 16, 1024), sdesc(k_s + kk * 32, 16, 1024), IDESC_QK8P, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)   // rope: 64 B a row
              mma_f8_ss_pair(d, sdesc(q_s + EQN_BYTES + kk * 32, 16, 512, kSwizzle64),
                             sdesc(k_s + EKN_BYTES + kk * 32, 16, 512, kSwizzle64), IDESC_QK8P, 1);
            tc_commit_pair(smem_u32(&sh->s_full[gj & 1]), kBoth);
            tc_commit_pair(smem_u32(&sh->k_empty[ks]), kBoth);
            if (j == it.n_kv - 1) tc_commit_pair(smem_u32(&sh->q_free[it_n & 1]), kBoth);
            return true;
          };
          auto issue_pv = [&](int j) -> bool {
            const uint32_t gp = g + j;
            const int vs = gp % PNV;
            // V and the free O first: they are ready long before P as a rule,
            // and checking them after P would add their barrier round trips to
            // the hand-off from the softmax to P*V.
            if (!mbar_wait_cluster(smem_u32(&sh->v_full[vs]), (gp / PNV) & 1, status, abort_flag)) return false;
            if (j == 0 && it_n >= 1 &&
                !mbar_wait_cluster(smem_u32(&sh->o_free), (it_n - 1) & 1, status, abort_flag))
              return false;
            if (!mbar_wait_cluster(smem_u32(&sh->p_full[gp & 1]), (gp >> 1) & 1, status, abort_flag)) return false;
            tc_fence_after();
            const uint32_t v_s = smem_u32(smem + E_SMEM_V + vs * PV_BYTES);
            const uint32_t pa = tmem + P_TM_S + (gp & 1) * 128;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_f16_ts_pair(o_t, pa + kk * 8, sdesc(v_s + kk * 2048, PBLK, 1024), IDESC_PV16P, (j > 0 || kk > 0));
            tc_commit_pair(smem_u32(&sh->o_done[gp & 1]), kBoth);
            tc_commit_pair(smem_u32(&sh->v_empty[vs]), kBoth);
            return true;
          };
          bool ok = issue_s(0);
          if (ok && n > 1) ok = issue_s(1);
          for (int j = 0; j < n && ok; ++j) {
            ok = issue_pv(j);
            if (ok && j + 2 < n) ok = issue_s(j + 2);
          }
          if (!ok) break;
          g += n;
          ++it_n;
        }
        tc_commit_pair(smem_u32(&sh->drain), 1);
        volatile int never = 0;
        mbar_wait(smem_u32(&sh->drain), 0, status, &never);
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------------- relay (CTA 1)
      // Forward "my half of K_j / V_j has landed" to CTA 0's ring barriers in
      // the order CTA 0's MMAs consume them: K_0, K_1, then V_j, K_{j+2}.
      if (elect_one()) {
        const uint32_t k_full0 = cluster_addr(smem_u32(&sh->k_full[0]), 0);
        const uint32_t v_full0 = cluster_addr(smem_u32(&sh->v_full[0]), 0);
        uint32_t g = 0;
        PairItem it;
        auto relay_k = [&](uint32_t gj) -> bool {
          const int ks = gj % PNK;
          if (!mbar_wait(smem_u32(&sh->k_full[ks]), (gj / PNK) & 1, status, abort_flag)) return false;
          mbar_arrive_cluster(k_full0 + ks * 8);
          return true;
        };
        auto relay_v = [&](uint32_t gj) -> bool {
          const int vs = gj % PNV;
          if (!mbar_wait(smem_u32(&sh->v_full[vs]), (gj / PNV) & 1, status, abort_flag)) return false;
          mbar_arrive_cluster(v_full0 + vs * 8);
          return true;
        };
        for (int idx = pair_id; next_pair(p, idx, n_pairs, total, rank, it, wl); idx += n_pairs) {
          const int n = it.n_kv;
          bool ok = relay_k(g);
          if (ok && n > 1) ok = relay_k(g + 1);
          for (int j = 0; j < n && ok; ++j) {
            ok = relay_v(g + j);
            if (ok && j + 2 < n) ok = relay_k(g + j + 2);
          }
          if (!ok) break;
          g += n;
        }
      }
      __syncwarp();
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ softmax + epilogue
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    const float sl2 = p.scale_log2;
    const float2 sl2v = make_float2(sl2, sl2);
    const uint32_t q_ready0 = cluster_addr(smem_u32(&sh->q_ready), 0);
    const uint32_t p_full0 = cluster_addr(smem_u32(&sh->p_full[0]), 0);
    const uint32_t o_free0 = cluster_addr(smem_u32(&sh->o_free), 0);
    uint32_t g = 0, it_n = 0;
    bool ok = true;

    // Item n's Q (read by the MMAs from shared memory) has landed in this CTA.
    auto stage_q = [&](uint32_t n) -> bool {
      if (!mbar_wait_warp(smem_u32(&sh->q_full[n & 1]), (n >> 1) & 1, status, abort_flag)) return false;
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(q_ready0);
      return true;
    };

    int idx = pair_id;
    PairItem it;
    bool have = next_pair(p, idx, n_pairs, total, rank, it, wl);
    if (have) ok = stage_q(0);
    while (have && ok) {
      const Item& own = it.own;
      const long long qpos = static_cast<long long>(own.cb) + own.i0 + row;
      const long long lim_all = min(static_cast<long long>(own.n_cb), qpos - own.co + 1);
      float m_run = kNegInf, l_run = 0.f;
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t gj = g + j;
        const uint32_t sb = gj & 1;
        if (!(ok = mbar_wait_cluster_warp(smem_u32(&sh->s_full[sb]), (gj >> 1) & 1, status, abort_flag))) break;
        tc_fence_after();
        float x[BN];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tmem + lane_off + P_TM_S + sb * 128 + c * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(reinterpret_cast<uint32_t*>(x) + c * 32));
        tmem_ld_wait();
        const long long lim = lim_all - static_cast<long long>(j) * BN;
        if (lim < BN) {
#pragma unroll
          for (int k = 0; k < BN; ++k) x[k] = k < lim ? x[k] : kNegInf;
        }
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmax3(x[i], x[8 + i], x[16 + i]);
#pragma unroll
        for (int k = 24; k + 16 <= BN; k += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], x[k + i], x[k + 8 + i]);
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], x[BN - 8 + i]);
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7]));
        const float m_new = fmaxf(m_run, mx * sl2);
        const bool need = m_new > m_run + kRescaleThreshold;
        const float f = need ? ex2(m_run - m_new) : 1.0f;
        if (need) m_run = m_new;
        const float msub = m_run == kNegInf ? 0.f : m_run;
        const float2 negm = make_float2(-msub, -msub);
        uint32_t pk[BN / 2];
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int k = 0; k < BN / 2; ++k) {
          const float2 t = __ffma2_rn(make_float2(x[2 * k], x[2 * k + 1]), sl2v, negm);
          const float2 e = make_float2(ex2(t.x), ex2(t.y));
          acc[k & 3] = __fadd2_rn(acc[k & 3], e);
          pk[k] = pack_f16(e.x, e.y);
        }
        const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
        const float2 a = __fadd2_rn(a01, a23);
        l_run = l_run * f + (a.x + a.y);
        if (j == it.n_kv - 1 && own.n_cb - j * BN < BN) {
          // Keys past the sequence in the last tile: zero this CTA's half of
          // those V rows (stale or non-finite) before P*V reads them.
          const int vs = gj % PNV;
          if (!(ok = mbar_wait_cluster_warp(smem_u32(&sh->v_full[vs]), (gj / PNV) & 1, status, abort_flag))) break;
          if (j * BN + row >= own.n_cb) {
            uint8_t* vrow = smem + E_SMEM_V + vs * PV_BYTES + row * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) reinterpret_cast<uint4*>(vrow)[c] = make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
        }
        tmem_st64(tmem + lane_off + P_TM_S + sb * 128, pk);
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // Rescale O only when the row maximum grew by more than 2^8, once P*V
          // of the previous tile has completed.
          if (!(ok = mbar_wait_cluster_warp(smem_u32(&sh->o_done[(gj - 1) & 1]), ((gj - 1) >> 1) & 1, status,
                                            abort_flag)))
            break;
          {
            tc_fence_after();
            uint32_t r[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t ta = tmem + lane_off + P_TM_O + c * 32;
              tmem_ld32(ta, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
              tmem_st32(ta, r);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(p_full0 + sb * 8);
      }
      if (!ok) break;
      g += it.n_kv;
      int nidx = idx + n_pairs;
      PairItem nx;
      const bool have_next = next_pair(p, nidx, n_pairs, total, rank, nx, wl);
      if (have_next && !(ok = stage_q(it_n + 1))) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = mbar_wait_cluster_warp(smem_u32(&sh->o_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, status,
                                        abort_flag)))
        break;
      tc_fence_after();
      float o[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld32(tmem + lane_off + P_TM_O + c * 32,
                  *reinterpret_cast<uint32_t(*)[32]>(reinterpret_cast<uint32_t*>(o) + c * 32));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(o_free0);
      const Item cur = it.own;
      it = nx;
      idx = nidx;
      have = have_next;
      ++it_n;
      store_row(p, cur, row, qpos, m_run, l_run, o);
    }
    // The completion of the P*V before the last (the other o_done barrier)
    // has arrived too: no asynchronous arrival may reach a CTA that has left.
    if (ok && g >= 2)
      mbar_wait_cluster_warp(smem_u32(&sh->o_done[(g - 2) & 1]), ((g - 2) >> 1) & 1, status, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // neither CTA frees TMEM or leaves while the pair still uses it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, P_TMEM_COLS);
  }
}

}  // namespace

// Two-CTA clusters of `kernel` (with `smem` bytes) that can be resident at
// once, per device (0 if none).
// Dynamic shared memory of a launch: the tiles and barriers, the compaction
// counts and a unit list as long as the chunk can need (the kernels walk all
// units without a list past kMaxUnits).
static int pair_smem_bytes(int units_offset, const Params& p) {
  const int n_units = ((p.n_qtiles + 1) >> 1) * p.B;
  const int listed = n_units <= kMaxUnits ? n_units : 0;
  return units_offset + 32 + 4 * listed + 1024;
}

// Two-CTA clusters of `kernel` (with `smem` bytes) that the current device can
// keep resident at once, or 0 if the query fails or none fits.
template <typename Kernel>
static int pair_clusters_of(Kernel kernel, int smem, int device, int slot) {
  static std::mutex mu;
  static int cached[4][64];
  static bool done[4][64];
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return 0;
  if (!done[slot][device]) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(P_THREADS);
    cfg.dynamicSmemBytes = smem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cached[slot][device] = n;
    done[slot][device] = true;
  }
  return cached[slot][device];
}
static int pair_clusters(int device, bool paged) {
  return paged ? pair_clusters_of(attn_pair_kernel<true>, P_SMEM_TOTAL, device, 2)
               : pair_clusters_of(attn_pair_kernel<false>, P_SMEM_TOTAL, device, 0);
}
static int pair_clusters_e4m3(int device, bool paged) {
  return paged ? pair_clusters_of(attn_pair_kernel_e4m3<true>, E_SMEM_TOTAL, device, 3)
               : pair_clusters_of(attn_pair_kernel_e4m3<false>, E_SMEM_TOTAL, device, 1);
}

cudaError_t launch_attention_pair(const AttnArgs& a, cudaStream_t stream) {
  const uint64_t HN = static_cast<uint64_t>(a.H) * 128;
  const uint64_t QW = static_cast<uint64_t>(a.H) * 192;
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap maps[4];
  const bool paged = a.kv_cache != nullptr;
  const uint64_t cache_rows = static_cast<uint64_t>(a.num_cache_rows);
  const bool ok = encode_2d(&maps[0], a.q, dt, QW, a.T_q, QW * 2, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) &&
                  encode_2d(&maps[1], a.k_nope, dt, HN, a.S, HN * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
                  (paged ? encode_2d(&maps[2], a.kv_cache, dt, 576, cache_rows, 1152, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B)
                         : encode_2d(&maps[2], a.k_rope, dt, 64, a.S, 128, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)) &&
                  encode_2d(&maps[3], a.v, dt, HN, a.S, HN * 2, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  Params p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.o_acc = a.o_acc;
  p.lse_acc = a.lse_acc;
  p.iro = a.iro;
  p.cache_len = a.cache_len;
  p.bro = a.bro;
  p.co = a.co;
  p.bl = a.bl;
  p.chunk = a.chunk;
  p.B = a.B;
  p.H = a.H;
  p.n_qtiles = (a.max_prompt_len + BM - 1) / BM;
  // Heads per group: about 16 MB of K_nope + V (bf16) in L2 (8 heads at 4096
  // buffer rows; 32 MB measured 1 % slower at the V3 shape and 3 % on a full
  // 8192-row chunk, 8 MB and less slower still).
  p.head_group = static_cast<int>(std::max<uint64_t>(1, (16ull << 20) / (static_cast<uint64_t>(a.S) * 512)));
  if (p.head_group > a.H) p.head_group = a.H;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.v_scale = a.v_scale;
  p.status = a.status;
  p.T_q = a.T_q;
  const PagedRope pr{static_cast<const uint8_t*>(a.kv_cache), a.cache_rows, a.num_cache_rows,
                     a.dtype == MLA_E4M3 ? 576 : 1152};
  const long long total = static_cast<long long>((p.n_qtiles + 1) / 2) * a.B * a.H;
  if (total <= 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int clusters = pair_clusters(dev, paged);
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  const int grid = 2 * static_cast<int>(total < clusters ? total : clusters);
  const int smem = pair_smem_bytes(P_SMEM_UNITS, p);
  if (paged)
    return launch_pdl(attn_pair_kernel<true>, dim3(grid), dim3(P_THREADS), smem, stream, maps[0], maps[1], maps[2],
                      maps[3], p, static_cast<int>(total), pr);
  else
    return launch_pdl(attn_pair_kernel<false>, dim3(grid), dim3(P_THREADS), smem, stream, maps[0], maps[1],
                      maps[2], maps[3], p, static_cast<int>(total), pr);
  return cudaGetLastError();
}

cudaError_t launch_attention_pair_e4m3(const AttnArgs& a, cudaStream_t stream) {
  const uint64_t HN = static_cast<uint64_t>(a.H) * 128;
  const uint64_t QW = static_cast<uint64_t>(a.H) * 192;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUtensorMap maps[5];
  const bool ok =
      encode_2d(&maps[0], a.q, u8, QW, a.T_q, QW, 128, BM, CU_TENSOR_MAP_SWIZZLE_128B) &&    // Q nope
      encode_2d(&maps[1], a.q, u8, QW, a.T_q, QW, 64, BM, CU_TENSOR_MAP_SWIZZLE_64B) &&      // Q rope
      encode_2d(&maps[2], a.k_nope, u8, HN, a.S, HN, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
      (a.kv_cache != nullptr
           ? encode_2d(&maps[3], a.kv_cache, u8, 576, static_cast<uint64_t>(a.num_cache_rows), 576, 64, 1,
                       CU_TENSOR_MAP_SWIZZLE_64B)
           : encode_2d(&maps[3], a.k_rope, u8, 64, a.S, 64, 64, 64, CU_TENSOR_MAP_SWIZZLE_64B)) &&
      encode_2d(&maps[4], a.v, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, HN, a.S, HN * 2, 64, BN,
                CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  Params p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.o_acc = a.o_acc;
  p.lse_acc = a.lse_acc;
  p.iro = a.iro;
  p.cache_len = a.cache_len;
  p.bro = a.bro;
  p.co = a.co;
  p.bl = a.bl;
  p.chunk = a.chunk;
  p.B = a.B;
  p.H = a.H;
  p.n_qtiles = (a.max_prompt_len + BM - 1) / BM;
  // Heads per group: about 32 MB of K_nope (e4m3) + V (f16) in L2.
  p.head_group = static_cast<int>(std::max<uint64_t>(1, (32ull << 20) / (static_cast<uint64_t>(a.S) * 384)));
  if (p.head_group > a.H) p.head_group = a.H;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.v_scale = a.v_scale;
  p.status = a.status;
  p.T_q = a.T_q;
  const PagedRope pr{static_cast<const uint8_t*>(a.kv_cache), a.cache_rows, a.num_cache_rows,
                     a.dtype == MLA_E4M3 ? 576 : 1152};
  const long long total = static_cast<long long>((p.n_qtiles + 1) / 2) * a.B * a.H;
  if (total <= 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool paged = a.kv_cache != nullptr;
  const int clusters = pair_clusters_e4m3(dev, paged);
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  const int grid = 2 * static_cast<int>(total < clusters ? total : clusters);
  const int smem = pair_smem_bytes(E_SMEM_UNITS, p);
  if (paged)
    return launch_pdl(attn_pair_kernel_e4m3<true>, dim3(grid), dim3(P_THREADS), smem, stream, maps[0], maps[1],
                      maps[2], maps[3], maps[4], p, static_cast<int>(total), pr);
  else
    return launch_pdl(attn_pair_kernel_e4m3<false>, dim3(grid), dim3(P_THREADS), smem, stream, maps[0], maps[1],
                      maps[2], maps[3], maps[4], p, static_cast<int>(total), pr);
  return cudaGetLastError();
}

// The one attention entry of the library: bf16 on the pair kernel, e4m3 on
// its e4m3 form.  A device that cannot keep a two-CTA cluster of the kernel
// resident gets an error (there is no other kernel to fall back to).
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  return a.dtype == MLA_E4M3 ? launch_attention_pair_e4m3(a, stream) : launch_attention_pair(a, stream);
}

}  // namespace mla
