// MLA prefill attention for one plan chunk ("flare_mla_prefill_dispatch":
// q [tokens, H, 192], ragged k (nope) and v [rows, H, 128], k_rope [rows, 64]
// shared by all heads, valid_length row offsets, scale, cache_offsets), with a
// causal mask offset by each sequence's cache length and a log-sum-exp merge
// of per-chunk results.
//
// Work item = (sequence b, 128-row query tile, head h).  Persistent CTAs (one
// per SM) stride over the items: heads in groups (so the CTAs in flight share
// a few heads' K/V in L2), heaviest query tiles first within a group.
//
//   warp 0      TMA producer of the Q tile (3 x 16 KB) and the K tiles (nope
//               2 x 16 KB + rope 16 KB), 128-byte swizzled, 2-stage K ring.
//   warp 6      TMA producer of the V tiles (2 x 16 KB), 2-stage V ring; kept
//               apart from K so K tiles run ahead of the V stages' release.
//   warp 1      TMEM owner (512 columns) and single-thread MMA issuer:
//                 S_j = Q K_j^T   M=128 queries, N=128 keys, K=192 as 12 MMAs;
//                                 A = Q read from tensor memory, B = K (K-major)
//                 O  += P_j V_j   M=128, N=128 (dv), K=128 keys as 8 MMAs;
//                                 A = P read from tensor memory, B = V (MN-major)
//               Keeping both A operands in TMEM leaves shared-memory bandwidth
//               to the K/V operands and the TMA writes.
//   warps 2..5  one thread per query row.  Copy the item's Q row from shared
//               memory into TMEM; per key tile: tcgen05.ld the S row, mask the
//               boundary tiles, row max, exp2 of s*scale*log2(e) - m with packed
//               f32x2 FMAs, row sum, bf16 P written back over S; O rescaled in
//               TMEM only when the row max grows by more than 2^8.  After the
//               last tile the next item's Q goes into TMEM (so its first MMAs
//               overlap this epilogue), then O / l, the natural-log LSE, and the
//               merge with earlier chunks (fp32 scratch) or the bf16 store.
//
// TMEM columns: S/P buffers 0..127 and 128..255, O 256..383, Q 384..479.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "attn_common.cuh"

namespace mla {
namespace {

constexpr int BLK = 128 * 128;                // one 128-row x 128-byte swizzled block
constexpr int Q_BYTES = 3 * BLK;              // 192 bf16 columns
constexpr int K_BYTES = 3 * BLK;              // nope 128 + rope 64
constexpr int V_BYTES = 2 * BLK;              // 128 dv
constexpr int NK = 2, NV = 2;
constexpr int SMEM_Q = 0;
constexpr int SMEM_K = SMEM_Q + Q_BYTES;
constexpr int SMEM_V = SMEM_K + NK * K_BYTES;
constexpr int SMEM_BAR = SMEM_V + NV * V_BYTES;   // 212992
constexpr int SMEM_UNITS = SMEM_BAR + 256;        // compaction counts, then the unit list
constexpr int SMEM_TOTAL = SMEM_UNITS + 32 + 4 * 4096 + 1024;   // the largest launch
constexpr int NUM_THREADS = 224;   // 7 warps: Q/K producer, MMA, 4 softmax, V producer
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;      // S/P buffers: columns 0..127, 128..255
constexpr uint32_t TM_O = 256;    // O: columns 256..383
constexpr uint32_t TM_Q = 384;    // Q (bf16 pairs): columns 384..479
constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16(BM, 128, false, true);

struct Smem {
  uint64_t q_full, q_empty, q_ready;
  uint64_t k_full[NK], k_empty[NK];
  uint64_t v_full[NV], v_empty[NV];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done[2], o_free;   // o_done[t & 1] completes when P*V of tile t does
  uint64_t drain;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(Smem) <= 256, "barrier block");

// Item order: heads in groups of `head_group`; within a group, query tiles
// heaviest first, and the group's heads side by side.  The CTAs in flight then
// share the K/V of a few heads in L2 instead of streaming every head's K/V.
// The units (sequence b, query tile qt) are those of the chunk with work,
// compacted in shared memory by every CTA first (up to kMaxUnits; beyond that
// all units are walked and the empty ones skipped), so that the static stride
// walks consecutive work and the CTAs in flight stay within one head group.
constexpr int kMaxUnits = 4096;

struct WorkList {
  const uint32_t* units;   // shared memory
  int n;                   // units with work, or -1: walk all units
};

__device__ __forceinline__ bool load_item(const Params& p, int idx, Item& it, const WorkList& wl) {
  const int n_units = wl.n >= 0 ? wl.n : p.n_qtiles * p.B;
  const int per_group = p.head_group * n_units;
  const int grp = idx / per_group;
  const int r = idx - grp * per_group;
  const int hg = min(p.head_group, p.H - grp * p.head_group);   // heads in this group
  const int ui = r / hg;
  const int h = grp * p.head_group + (r - ui * hg);
  const int unit = wl.n >= 0 ? static_cast<int>(wl.units[ui]) : ui;
  const int qt = p.n_qtiles - 1 - unit / p.B;   // heaviest query tiles first
  return tile_item(p, unit % p.B, h, qt, it);
}

// First item with work at or after `idx` (stepping by the grid size).
__device__ __forceinline__ bool next_item(const Params& p, int& idx, int total, Item& it, const WorkList& wl) {
  for (; idx < total; idx += gridDim.x)
    if (load_item(p, idx, it, wl)) return true;
  return false;
}

// Every thread of the CTA: compact the units with work into `list`; returns
// their count (the same in every thread), or -1 past kMaxUnits.
__device__ int compact_units(const Params& p, uint32_t* list, int* warp_cnt) {
  const int n_units = p.n_qtiles * p.B;
  if (n_units > kMaxUnits) return -1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nwarps = static_cast<int>(blockDim.x) >> 5;
  int base = 0;
  for (int u0 = 0; u0 < n_units; u0 += static_cast<int>(blockDim.x)) {
    const int u = u0 + tid;
    bool has = false;
    if (u < n_units) {
      Item a;
      has = tile_item(p, u % p.B, 0, p.n_qtiles - 1 - u / p.B, a);
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

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap kn_map,
                const __grid_constant__ CUtensorMap kr_map, const __grid_constant__ CUtensorMap v_map,
                const Params p, int total_items) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Smem* sh = reinterpret_cast<Smem*>(smem + SMEM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (p.bl[p.chunk] <= 0) return;
  if (p.status && *reinterpret_cast<volatile int32_t*>(p.status) == MLA_DEV_TIMEOUT) return;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sh->q_full), 1);
    mbar_init(smem_u32(&sh->q_empty), 4);
    mbar_init(smem_u32(&sh->q_ready), 4);
    for (int i = 0; i < NK; ++i) {
      mbar_init(smem_u32(&sh->k_full[i]), 1);
      mbar_init(smem_u32(&sh->k_empty[i]), 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(smem_u32(&sh->v_full[i]), 1);
      mbar_init(smem_u32(&sh->v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh->s_full[i]), 1);
      mbar_init(smem_u32(&sh->p_full[i]), 4);
    }
    mbar_init(smem_u32(&sh->o_done[0]), 1);
    mbar_init(smem_u32(&sh->o_done[1]), 1);
    mbar_init(smem_u32(&sh->o_free), 4);
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sh->tmem), TMEM_COLS);
    tmem_relinquish();
  }
  // Compaction counts (8 ints), then the list, sized by the launch.
  const WorkList wl{reinterpret_cast<const uint32_t*>(smem + SMEM_UNITS + 32),
                    compact_units(p, reinterpret_cast<uint32_t*>(smem + SMEM_UNITS + 32),
                                  reinterpret_cast<int*>(smem + SMEM_UNITS))};
  const int total = wl.n >= 0 ? wl.n * p.H : total_items;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem;
  volatile int* abort_flag = &sh->abort;
  int32_t* status = p.status;

  if (warp == 0) {
    // ------------------------------------------------------------ Q and K producer
    // The whole warp runs the loop and waits; one elected lane issues copies.
    if (elect_one()) {
      prefetch_tmap(&q_map);
      prefetch_tmap(&kn_map);
      prefetch_tmap(&kr_map);
    }
    __syncwarp();
    uint32_t g = 0, it_n = 0;
    int q_last = -1, k_last[NK] = {-1, -1};
    bool ok = true;
    Item it;
    for (int idx = blockIdx.x; ok && next_item(p, idx, total, it, wl); idx += gridDim.x) {
      // The shared-memory Q buffer is free once the previous item's Q is in TMEM.
      if (it_n > 0 && !(ok = mbar_wait_warp(smem_u32(&sh->q_empty), (it_n - 1) & 1, status, abort_flag))) break;
      if (elect_one()) {
        const uint32_t qf = smem_u32(&sh->q_full);
        mbar_expect_tx(qf, Q_BYTES);
        for (int blk = 0; blk < 3; ++blk)
          tma_load_2d(smem_u32(smem + SMEM_Q + blk * BLK), &q_map, qf, it.h * 192 + blk * 64, it.q_row0);
      }
      __syncwarp();
      q_last = int(it_n & 1);
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t gj = g + j;
        const int row = it.kv_row0 + j * BN;
        const int ks = gj % NK;
        // K stage ks is free once S_{gj-2} (same stage, same S buffer) has
        // completed: s_full[ks] doubles as the stage's release.
        if (gj >= NK && !(ok = mbar_wait_warp(smem_u32(&sh->s_full[ks]), ((gj - NK) / NK) & 1, status, abort_flag))) break;
        if (elect_one()) {
          const uint32_t kf = smem_u32(&sh->k_full[ks]);
          mbar_expect_tx(kf, K_BYTES);
          const uint32_t kdst = smem_u32(smem + SMEM_K + ks * K_BYTES);
          tma_load_2d(kdst, &kn_map, kf, it.h * 128, row);
          tma_load_2d(kdst + BLK, &kn_map, kf, it.h * 128 + 64, row);
          tma_load_2d(kdst + 2 * BLK, &kr_map, kf, 0, row);
        }
        __syncwarp();
        k_last[ks] = int((gj / NK) & 1);
      }
      g += it.n_kv;
      ++it_n;
    }
    // Drain: every issued load lands before the CTA exits.
    volatile int never = 0;
    if (q_last >= 0) mbar_wait_warp(smem_u32(&sh->q_full), uint32_t(q_last), status, &never);
    for (int s = 0; s < NK; ++s)
      if (k_last[s] >= 0) mbar_wait_warp(smem_u32(&sh->k_full[s]), uint32_t(k_last[s]), status, &never);
  } else if (warp == 6) {
    // ------------------------------------------------------------ V producer
    // Separate from K so that K tiles run ahead of the V stages' release.
    if (elect_one()) prefetch_tmap(&v_map);
    __syncwarp();
    uint32_t g = 0;
    int v_last[NV] = {-1, -1};
    bool ok = true;
    Item it;
    for (int idx = blockIdx.x; ok && next_item(p, idx, total, it, wl); idx += gridDim.x) {
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t gj = g + j;
        const int row = it.kv_row0 + j * BN;
        const int vs = gj % NV;
        // V stage vs is free once P*V of tile gj-2 (same stage) has completed.
        // o_done[gj & 1] completes once per P*V of that parity; a P*V two
        // ahead on it would need this very V tile, so it cannot run ahead.
        if (gj >= NV && !(ok = mbar_wait_warp(smem_u32(&sh->o_done[gj & 1]), ((gj - NV) >> 1) & 1, status, abort_flag))) break;
        if (elect_one()) {
          const uint32_t vf = smem_u32(&sh->v_full[vs]);
          mbar_expect_tx(vf, V_BYTES);
          const uint32_t vdst = smem_u32(smem + SMEM_V + vs * V_BYTES);
          tma_load_2d(vdst, &v_map, vf, it.h * 128, row);
          tma_load_2d(vdst + BLK, &v_map, vf, it.h * 128 + 64, row);
        }
        __syncwarp();
        v_last[vs] = int((gj / NV) & 1);
      }
      g += it.n_kv;
    }
    volatile int never = 0;
    for (int s = 0; s < NV; ++s)
      if (v_last[s] >= 0) mbar_wait_warp(smem_u32(&sh->v_full[s]), uint32_t(v_last[s]), status, &never);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One elected lane runs the whole loop, waits included, and the warp
    // reconverges only at the end.  Reconverging a warp whose lane has MMAs in
    // flight stalls it until most of them have executed, and a wait that then
    // follows leaves the tensor pipe idle; a lone elected lane goes straight
    // from one MMA group to the next wait and back.
    if (elect_one()) {
      uint32_t g = 0, it_n = 0;
      const uint32_t q_t = tmem + TM_Q;
      const uint32_t o_t = tmem + TM_O;
      Item it;
      for (int idx = blockIdx.x; next_item(p, idx, total, it, wl); idx += gridDim.x) {
        if (!mbar_wait(smem_u32(&sh->q_ready), it_n & 1, status, abort_flag)) break;
        const int n = it.n_kv;
        // S_j = Q K_j^T into S buffer j % 2 (it last held P_{j-2}, whose P*V
        // was issued earlier; tcgen05 MMAs execute in issue order).
        auto issue_s = [&](int j) -> bool {
          const uint32_t gj = g + j;
          const int ks = gj % NK;
          if (!mbar_wait(smem_u32(&sh->k_full[ks]), (gj / NK) & 1, status, abort_flag)) return false;
          tc_fence_after();
          const uint32_t k_s = smem_u32(smem + SMEM_K + ks * K_BYTES);
          const uint32_t d = tmem + TM_S + (gj & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < 12; ++kk) {
            const uint32_t off = (kk >> 2) * BLK + (kk & 3) * 32;
            mma_f16_ts(d, q_t + kk * 8, sdesc(k_s + off, 16, 1024), IDESC_QK, kk > 0);
          }
          tc_commit(smem_u32(&sh->s_full[gj & 1]));
          return true;
        };
        // O += P_j V_j.
        auto issue_pv = [&](int j) -> bool {
          const uint32_t gp = g + j;
          const int vs = gp % NV;
          if (!mbar_wait(smem_u32(&sh->p_full[gp & 1]), (gp >> 1) & 1, status, abort_flag)) return false;
          if (!mbar_wait(smem_u32(&sh->v_full[vs]), (gp / NV) & 1, status, abort_flag)) return false;
          // The previous item's epilogue must have read O before it is overwritten.
          if (j == 0 && it_n >= 1 && !mbar_wait(smem_u32(&sh->o_free), (it_n - 1) & 1, status, abort_flag))
            return false;
          tc_fence_after();
          const uint32_t v_s = smem_u32(smem + SMEM_V + vs * V_BYTES);
          const uint32_t pa = tmem + TM_S + (gp & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_f16_ts(o_t, pa + kk * 8, sdesc(v_s + kk * 2048, BLK, 1024), IDESC_PV, (j > 0 || kk > 0));
          tc_commit(smem_u32(&sh->o_done[gp & 1]));
          return true;
        };
        // Two S tiles ahead; then each P_j*V_j as soon as P_j is ready,
        // followed by S_{j+2}.
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
      tc_commit(smem_u32(&sh->drain));
      volatile int never = 0;
      mbar_wait(smem_u32(&sh->drain), 0, status, &never);
    }
    __syncwarp();
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ softmax + epilogue
    const int q4 = warp & 3;                 // TMEM lane quarter
    const int row = q4 * 32 + lane;          // query row within the tile (= TMEM lane)
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    const float sl2 = p.scale_log2;
    const float2 sl2v = make_float2(sl2, sl2);
    uint32_t g = 0, it_n = 0;
    bool ok = true;

    // Item n's Q row: shared memory (after its TMA) -> registers -> TMEM, then
    // release the shared buffer and tell the MMA warp.
    auto stage_q = [&](uint32_t n) -> bool {
      if (!mbar_wait_warp(smem_u32(&sh->q_full), n & 1, status, abort_flag)) return false;
      uint32_t v[96];
      const uint8_t* qs = smem + SMEM_Q + row * 128;
#pragma unroll
      for (int j = 0; j < 24; ++j) {
        const uint4 x = *reinterpret_cast<const uint4*>(qs + (j >> 3) * BLK + (((j & 7) ^ (row & 7)) << 4));
        v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
      }
      tmem_st32(tmem + lane_off + TM_Q, v);
      tmem_st32(tmem + lane_off + TM_Q + 32, v + 32);
      tmem_st32(tmem + lane_off + TM_Q + 64, v + 64);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh->q_empty));
        mbar_arrive(smem_u32(&sh->q_ready));
      }
      return true;
    };

    int idx = blockIdx.x;
    Item it;
    bool have = next_item(p, idx, total, it, wl);
    if (have) ok = stage_q(0);
    while (have && ok) {
      const long long qpos = static_cast<long long>(it.cb) + it.i0 + row;
      // Relative key index kk is visible iff kk < lim_all.
      const long long lim_all = min(static_cast<long long>(it.n_cb), qpos - it.co + 1);
      float m_run = kNegInf, l_run = 0.f;
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t gj = g + j;
        const uint32_t sb = gj & 1;
        if (!(ok = mbar_wait_warp(smem_u32(&sh->s_full[sb]), (gj >> 1) & 1, status, abort_flag))) break;
        tc_fence_after();
        // Raw scores of this row: four TMEM loads in flight, one wait.
        float x[BN];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tmem + lane_off + TM_S + sb * 128 + c * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(reinterpret_cast<uint32_t*>(x) + c * 32));
        tmem_ld_wait();
        const long long lim = lim_all - static_cast<long long>(j) * BN;
        if (lim < BN) {
#pragma unroll
          for (int k = 0; k < BN; ++k) x[k] = k < lim ? x[k] : kNegInf;
        }
        // Row maximum: 3-input max over 8 independent chains.
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmax3(x[i], x[8 + i], x[16 + i]);
#pragma unroll
        for (int k = 24; k < BN; k += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], x[k + i], x[k + 8 + i]);
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7]));
        // Scores enter exp2 as s * scale*log2(e) - m (scale > 0, so the max
        // commutes with the scaling).
        const float m_new = fmaxf(m_run, mx * sl2);
        const bool need = m_new > m_run + kRescaleThreshold;
        const float f = need ? ex2(m_run - m_new) : 1.0f;   // m_run = -inf gives 0
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
        if (j == it.n_kv - 1 && it.n_cb - j * BN < BN) {
          // The last tile reaches past the sequence's keys: those V rows may hold
          // anything (even non-finite values), so zero them before P*V reads them.
          const int vs = gj % NV;
          if (!(ok = mbar_wait_warp(smem_u32(&sh->v_full[vs]), (gj / NV) & 1, status, abort_flag))) break;
          if (j * BN + row >= it.n_cb) {
            uint8_t* vrow = smem + SMEM_V + vs * V_BYTES + row * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              reinterpret_cast<uint4*>(vrow)[c] = make_uint4(0, 0, 0, 0);
              reinterpret_cast<uint4*>(vrow + BLK)[c] = make_uint4(0, 0, 0, 0);
            }
          }
          fence_async_smem();
        }
        tmem_st32(tmem + lane_off + TM_S + sb * 128, pk);
        tmem_st32(tmem + lane_off + TM_S + sb * 128 + 32, pk + 32);
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // The row maximum grew by more than 2^8: rescale O in TMEM once P*V
          // of the previous tile has completed, before P_j*V_j.  Otherwise P_j
          // goes out without that wait.  (The wait cannot alias a later phase:
          // the next P*V on the same barrier needs a P this warp has not
          // produced yet.)
          if (!(ok = mbar_wait_warp(smem_u32(&sh->o_done[(gj - 1) & 1]), ((gj - 1) >> 1) & 1, status, abort_flag))) break;
          {
            tc_fence_after();
            uint32_t r[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t ta = tmem + lane_off + TM_O + c * 32;
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
        if (lane == 0) mbar_arrive(smem_u32(&sh->p_full[sb]));
      }
      if (!ok) break;
      g += it.n_kv;
      // All of this item's S MMAs are done (the last one was waited for), so
      // its Q can be replaced: stage the next item's Q now, letting that
      // item's first MMAs run under this epilogue.
      int nidx = idx + gridDim.x;
      Item nx;
      const bool have_next = next_item(p, nidx, total, nx, wl);
      if (have_next && !(ok = stage_q(it_n + 1))) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = mbar_wait_warp(smem_u32(&sh->o_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, status, abort_flag))) break;
      tc_fence_after();
      float o[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld32(tmem + lane_off + TM_O + c * 32,
                  *reinterpret_cast<uint32_t(*)[32]>(reinterpret_cast<uint32_t*>(o) + c * 32));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->o_free));
      const Item cur = it;
      it = nx;
      idx = nidx;
      have = have_next;
      ++it_n;
      store_row(p, cur, row, qpos, m_run, l_run, o);
    }
    // The completion of the P*V before the last (the other o_done barrier)
    // has arrived too: no asynchronous arrival may reach a CTA that has left.
    if (ok && g >= 2)
      mbar_wait_warp(smem_u32(&sh->o_done[(g - 2) & 1]), ((g - 2) >> 1) & 1, status, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

// MLA_ATTENTION_KERNEL=single|pair picks the bf16 kernel (default: the two-SM
// pair kernel where the device can run it).
bool attention_uses_pair() {
  const char* v = std::getenv("MLA_ATTENTION_KERNEL");
  if (v != nullptr && std::strcmp(v, "single") == 0) return false;
  return attention_pair_available();
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  if (a.dtype == MLA_E4M3) return launch_attention_pair_e4m3(a, stream);
  if (attention_uses_pair()) return launch_attention_pair(a, stream);
  const uint64_t HN = static_cast<uint64_t>(a.H) * 128;
  const uint64_t QW = static_cast<uint64_t>(a.H) * 192;
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap maps[4];
  const bool ok = encode_2d(&maps[0], a.q, dt, QW, a.T_q, QW * 2, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) &&
                  encode_2d(&maps[1], a.k_nope, dt, HN, a.S, HN * 2, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B) &&
                  encode_2d(&maps[2], a.k_rope, dt, 64, a.S, 128, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B) &&
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
  // Heads per group: about 32 MB of K_nope + V (S rows x 512 B per head) in L2.
  p.head_group = static_cast<int>(std::max<uint64_t>(1, (32ull << 20) / (static_cast<uint64_t>(a.S) * 512)));
  if (p.head_group > a.H) p.head_group = a.H;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.v_scale = a.v_scale;
  p.status = a.status;
  const long long total = static_cast<long long>(p.n_qtiles) * a.B * a.H;
  if (total <= 0) return cudaSuccess;
  const int grid = total < sm_count() ? static_cast<int>(total) : sm_count();
  cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
  const int n_units = p.n_qtiles * p.B;
  const int smem_bytes = SMEM_UNITS + 32 + 4 * (n_units <= kMaxUnits ? n_units : 0) + 1024;
  attn_kernel<<<grid, NUM_THREADS, smem_bytes, stream>>>(maps[0], maps[1], maps[2], maps[3], p,
                                                        static_cast<int>(total));
  return cudaGetLastError();
}

}  // namespace mla
