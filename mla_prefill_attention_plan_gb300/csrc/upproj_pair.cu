// Up-projection on pairs of SMs ("mla_prefill_decode_graph_bf16", Args: w_k,
// w_uv): the GEMM  [rows, 512] x [512, 2*H*128]  of upproj.cu (N axis = the
// 128-wide head blocks of w_k then of w_uv), with 256 x 256 output tiles
// computed by a cluster of two CTAs through two-SM MMAs (cta_group::2,
// M = 256).  CTA r holds rows [128r, 128r + 128) of the tile's A and D, and
// B rows (N) [128r, 128r + 128) of the tile: each SM loads 32 KB per k-block
// for 128 x 256 x k of tensor work, against 48 KB in the one-SM kernel, whose
// L2 -> SM stream (~94 B/clk per SM at the tensor rate) exceeds what L2
// delivers to every SM at once (~72 B/clk).
//
//   warp 0      TMA producer: own A rows and own B half per k-block, 6-stage ring.
//               A comes from the chunk's c_kv buffer (one tile load), or
//               straight from the paged cache: the chunk's cache-row table
//               gives the tile's 128 rows (read a tile ahead), and per
//               k-block the warp copies the rows' 128-byte slices with
//               16-byte cp.async into the swizzled layout the tile load
//               would give.  A stage's
//               A rows are counted on its barrier A_LAG stages later, once
//               they have landed and been fenced into the async proxy.
//   warp 1      both CTAs: TMEM allocation (512 columns, pair form).
//               CTA 0: one elected lane issues the pair MMAs (M=256, N=256)
//               into one of two 256-column accumulators and commits to the
//               barriers of both CTAs.  CTA 1: one elected lane relays "my
//               k-block landed" to CTA 0's ring barriers.
//   warps 2..5  epilogue of the CTA's own 128 rows, as in upproj.cu; "this
//               accumulator has been read" goes to CTA 0.
#include <mutex>

#include "kernels.cuh"

namespace mla {
namespace {

constexpr int UBM = 128, UBN = 256, UBKB = 128;   // rows per CTA, tile cols, k-block bytes
constexpr int USTAGES = 6;
constexpr int UA_BYTES = UBM * UBKB;              // 16 KB: own A rows
constexpr int UB_BYTES = (UBN / 2) * UBKB;        // 16 KB: own half of B
constexpr int UEPI_BYTES = 32 * 128;
constexpr int U_SMEM_A = 0;
constexpr int U_SMEM_B = U_SMEM_A + USTAGES * UA_BYTES;
constexpr int U_SMEM_EPI = U_SMEM_B + USTAGES * UB_BYTES;          // 196608
constexpr int U_SMEM_BAR = U_SMEM_EPI + 4 * 2 * UEPI_BYTES;        // 229376
constexpr int U_SMEM_TOTAL = U_SMEM_BAR + 256 + 1024;
constexpr int U_THREADS = 192;
constexpr uint32_t U_TMEM_COLS = 512;
constexpr uint16_t kPairMask = 3;

struct PairGemmSmem {
  uint64_t full[USTAGES];    // CTA 0: own bytes + the relay; CTA 1: own bytes
  uint64_t empty[USTAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];        // CTA 0: both CTAs' epilogues (8 warps)
  uint64_t drain;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(PairGemmSmem) <= 256, "barrier block");

// Where the A rows live when they are read from the paged cache.
struct PagedA {
  const uint8_t* cache;       // cache rows of row_bytes; c_kv = the first 512 * ELT bytes of a row
  const int32_t* rows;        // the chunk's cache row of each buffer row, or null: A is the c_kv buffer
  int num_rows, row_bytes;
};
// Stages between a stage's A copies and its arrival (cp.async groups left
// pending): enough to cover the copies' latency at the tensor rate, fewer
// than the ring's stages.
constexpr int A_LAG = 4;
static_assert(A_LAG < USTAGES, "the ring must hold the lagging stages");

// Stage `bar`'s A copies have landed (all but the newest N cp.async groups
// of the warp): fence them into the async proxy, count them on the barrier.
template <int N>
__device__ __forceinline__ void a_rows_landed(uint32_t bar) {
  cp_async_wait<N>();
  fence_async_smem();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// PAGED: A rows from the paged cache through the chunk's cache-row table (an
// instantiation of its own, so that the buffered one carries no trace of it).
template <int ELT, bool PAGED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(U_THREADS, 1)
    upproj_pair_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap wk_map,
                       const __grid_constant__ CUtensorMap wuv_map,
                       const __grid_constant__ CUtensorMap k_out_map,
                       const __grid_constant__ CUtensorMap v_out_map, const int32_t* buffer_lengths,
                       int chunk, int S, int H, float out_scale, int32_t* status, const PagedA pa) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairGemmSmem* sh = reinterpret_cast<PairGemmSmem*>(smem + U_SMEM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair_id = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;

  pdl_enter();
  // Both CTAs of a pair read the same row count, so they return together.
  int rows = buffer_lengths ? buffer_lengths[chunk] : S;
  if (rows <= 0) return;
  if (rows > S) rows = S;
  const int num_m = (rows + 2 * UBM - 1) / (2 * UBM);   // 256-row pair tiles
  constexpr int KB = 512 * ELT / UBKB;                  // k-blocks: 8 (bf16) or 4 (e4m3)
  constexpr int KSTEP = 32;                             // bytes of one MMA's K
  constexpr uint32_t IDESC = ELT == 2 ? idesc_bf16(2 * UBM, UBN, false, false) : idesc_e4m3(2 * UBM, UBN, false, false);

  if (threadIdx.x == 0) {
    const uint32_t lead = rank == 0 ? 1u : 0u;
    for (int s = 0; s < USTAGES; ++s) {
      // own bytes (+ the paged A rows) + in CTA 0 the relay
      mbar_init(smem_u32(&sh->full[s]), 1 + lead + (PAGED ? 1u : 0u));
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh->tfull[i]), 1);
      mbar_init(smem_u32(&sh->tempty[i]), 8);
    }
    mbar_init(smem_u32(&sh->drain), 1);
    // A pipeline timeout recorded by an earlier kernel on this status word:
    // do no work (the pair agrees through cluster_any below).
    sh->abort = timed_out_before(status) ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&sh->tmem), U_TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const int num_tiles = cluster_any(&sh->abort) ? 0 : num_m * H;   // N: 2*H*128 / 256
  const uint32_t tmem = sh->tmem;
  volatile int* abort_flag = &sh->abort;

  if (warp == 0) {
    if constexpr (!PAGED) {
      // One lane issues both tile loads of every k-block.
      if (lane == 0) {
        prefetch_tmap(&a_map);
        prefetch_tmap(&wk_map);
        prefetch_tmap(&wuv_map);
        int stage = 0;
        uint32_t phase = 0;
        int last_ph[USTAGES];
        for (int s = 0; s < USTAGES; ++s) last_ph[s] = -1;
        for (int t = pair_id; t < num_tiles && !*abort_flag; t += n_pairs) {
          const int m0 = (t % num_m) * 2 * UBM + static_cast<int>(rank) * UBM;
          const int nt = t / num_m;
          const int hf = 2 * nt + static_cast<int>(rank);   // this CTA's 128-wide block of N
          const CUtensorMap* wmap = hf < H ? &wk_map : &wuv_map;
          bool ok = true;
          for (int kb = 0; kb < KB; ++kb) {
            if (!(ok = mbar_wait(smem_u32(&sh->empty[stage]), phase ^ 1, status, abort_flag))) break;
            const uint32_t full = smem_u32(&sh->full[stage]);
            mbar_expect_tx(full, UA_BYTES + UB_BYTES);
            const int x = kb * (UBKB / ELT);
            tma_load_2d(smem_u32(smem + U_SMEM_A + stage * UA_BYTES), &a_map, full, x, m0);
            tma_load_2d(smem_u32(smem + U_SMEM_B + stage * UB_BYTES), wmap, full, x, (hf % H) * 128);
            last_ph[stage] = int(phase);
            if (++stage == USTAGES) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
        }
        volatile int never = 0;
        for (int s = 0; s < USTAGES; ++s)
          if (last_ph[s] >= 0) mbar_wait(smem_u32(&sh->full[s]), uint32_t(last_ph[s]), status, &never);
        // ... and every stage release the MMAs committed to this CTA has
        // arrived: an asynchronous arrival must not reach a CTA that has left.
        for (int s = 0; s < USTAGES; ++s)
          if (last_ph[s] >= 0) mbar_wait(smem_u32(&sh->empty[s]), uint32_t(last_ph[s]), status, abort_flag);
      }
    } else {
      // The whole warp runs the loop: every lane issues A copies.
      if (lane == 0) {
        prefetch_tmap(&a_map);
        prefetch_tmap(&wk_map);
        prefetch_tmap(&wuv_map);
      }
      int stage = 0;
      uint32_t phase = 0;
      int last_ph[USTAGES];
      for (int s = 0; s < USTAGES; ++s) last_ph[s] = -1;
      int issued = 0;   // stages whose A copies were issued (the last A_LAG not yet counted)
      // Paged A: the cache rows of the tile's rows 4 lane .. 4 lane + 3, loaded
      // a tile ahead of their use (0 past the chunk's rows).
      int yn[4] = {0, 0, 0, 0};
      auto fetch_rows = [&](int t) {
        const int m0 = (t % num_m) * 2 * UBM + static_cast<int>(rank) * UBM;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = m0 + 4 * lane + k;
          yn[k] = t < num_tiles && r < rows ? __ldg(pa.rows + r) : 0;
        }
      };
      fetch_rows(pair_id);
      for (int t = pair_id; t < num_tiles && !__any_sync(0xffffffffu, *abort_flag != 0); t += n_pairs) {
        const int m0 = (t % num_m) * 2 * UBM + static_cast<int>(rank) * UBM;
        const int nt = t / num_m;
        const int hf = 2 * nt + static_cast<int>(rank);   // this CTA's 128-wide block of N
        const CUtensorMap* wmap = hf < H ? &wk_map : &wuv_map;
        // Paged A: lane l copies 16-byte chunk l % 8 of tile rows 4i + l / 8
        // (i < 32); arow[i] is that row's cache row.  Row 4i + k is lane i's
        // k-th row.  A row outside the cache is reported and read as row 0.
        int arow[32];
        {
          int y[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) y[k] = yn[k];
          fetch_rows(t + n_pairs);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (static_cast<unsigned>(y[k]) >= static_cast<unsigned>(pa.num_rows)) {
              set_status(status, MLA_DEV_BAD_PAGE);
              y[k] = 0;
            }
          }
          const int k = lane >> 3;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int v0 = __shfl_sync(0xffffffffu, y[0], i), v1 = __shfl_sync(0xffffffffu, y[1], i);
            const int v2 = __shfl_sync(0xffffffffu, y[2], i), v3 = __shfl_sync(0xffffffffu, y[3], i);
            arow[i] = k == 0 ? v0 : k == 1 ? v1 : k == 2 ? v2 : v3;
          }
        }
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!(ok = mbar_wait_warp(smem_u32(&sh->empty[stage]), phase ^ 1, status, abort_flag))) break;
          const uint32_t full = smem_u32(&sh->full[stage]);
          const uint32_t adst = smem_u32(smem + U_SMEM_A + stage * UA_BYTES);
          const int x = kb * (UBKB / ELT);
          if (elect_one()) {
            mbar_expect_tx(full, UB_BYTES);
            tma_load_2d(smem_u32(smem + U_SMEM_B + stage * UB_BYTES), wmap, full, x, (hf % H) * 128);
          }
          __syncwarp();
          {
            const int c = lane & 7;
            const uint8_t* src = pa.cache + kb * UBKB + c * 16;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int r = 4 * i + (lane >> 3);
              cp_async16(adst + r * UBKB + ((c ^ (r & 7)) << 4), src + static_cast<size_t>(arow[i]) * pa.row_bytes);
            }
            cp_async_commit();
            if (++issued > A_LAG) {
              const int ls = (stage + USTAGES - A_LAG) % USTAGES;
              a_rows_landed<A_LAG>(smem_u32(&sh->full[ls]));
            }
          }
          last_ph[stage] = int(phase);
          if (++stage == USTAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
      // The last stages' A rows (at most A_LAG), oldest first.
      {
        cp_async_wait<0>();
        fence_async_smem();
        __syncwarp();
        const int n = issued < A_LAG ? issued : A_LAG;
        if (lane == 0)
          for (int j = n; j >= 1; --j) mbar_arrive(smem_u32(&sh->full[(stage + USTAGES - j) % USTAGES]));
        __syncwarp();
      }
      if (lane == 0) {
        volatile int never = 0;
        for (int s = 0; s < USTAGES; ++s)
          if (last_ph[s] >= 0) mbar_wait(smem_u32(&sh->full[s]), uint32_t(last_ph[s]), status, &never);
        // ... and every stage release the MMAs committed to this CTA has
        // arrived: an asynchronous arrival must not reach a CTA that has left.
        for (int s = 0; s < USTAGES; ++s)
          if (last_ph[s] >= 0) mbar_wait(smem_u32(&sh->empty[s]), uint32_t(last_ph[s]), status, abort_flag);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // One elected lane runs the whole issue loop (no reconvergence while
      // MMAs are in flight).
      if (elect_one()) {
        int stage = 0;
        uint32_t phase = 0;
        int tl = 0;
        bool ok = true;
        for (int t = pair_id; t < num_tiles && ok; t += n_pairs, ++tl) {
          const int acc = tl & 1;
          if (!(ok = mbar_wait(smem_u32(&sh->tempty[acc]), ((tl >> 1) & 1) ^ 1, status, abort_flag))) break;
          tc_fence_after();
          const uint32_t d = tmem + acc * UBN;
          for (int kb = 0; kb < KB; ++kb) {
            if (!(ok = mbar_wait(smem_u32(&sh->full[stage]), phase, status, abort_flag))) break;
            tc_fence_after();
            const uint32_t a = smem_u32(smem + U_SMEM_A + stage * UA_BYTES);
            const uint32_t b = smem_u32(smem + U_SMEM_B + stage * UB_BYTES);
#pragma unroll
            for (int k = 0; k < UBKB / KSTEP; ++k) {
              const uint64_t ad = sdesc(a + k * KSTEP, 16, 1024);
              const uint64_t bd = sdesc(b + k * KSTEP, 16, 1024);
              if (ELT == 2) mma_f16_ss_pair(d, ad, bd, IDESC, (kb | k) != 0);
              else mma_f8_ss_pair(d, ad, bd, IDESC, (kb | k) != 0);
            }
            tc_commit_pair(smem_u32(&sh->empty[stage]), kPairMask);
            if (++stage == USTAGES) { stage = 0; phase ^= 1; }
          }
          if (ok) tc_commit_pair(smem_u32(&sh->tfull[acc]), kPairMask);
        }
        tc_commit_pair(smem_u32(&sh->drain), 1);
        volatile int never = 0;
        mbar_wait(smem_u32(&sh->drain), 0, status, &never);
      }
      __syncwarp();
    } else {
      // Relay: CTA 1's k-blocks to CTA 0's ring, in order.
      if (elect_one()) {
        const uint32_t full0 = cluster_addr(smem_u32(&sh->full[0]), 0);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = pair_id; t < num_tiles && ok; t += n_pairs) {
          for (int kb = 0; kb < KB; ++kb) {
            if (!(ok = mbar_wait(smem_u32(&sh->full[stage]), phase, status, abort_flag))) break;
            mbar_arrive_cluster(full0 + stage * 8);
            if (++stage == USTAGES) { stage = 0; phase ^= 1; }
          }
        }
      }
      __syncwarp();
    }
  } else {
    // Epilogue warps 2..5: TMEM lane quarter q = warp % 4 holds rows 32q..32q+31.
    const int q = warp & 3;
    const uint32_t lane_off = uint32_t(q * 32) << 16;
    const uint32_t tempty0 = cluster_addr(smem_u32(&sh->tempty[0]), 0);
    uint8_t* stage_buf = smem + U_SMEM_EPI + (warp - 2) * 2 * UEPI_BYTES;
    int buf = 0;
    int tl = 0;
    for (int t = pair_id; t < num_tiles; t += n_pairs, ++tl) {
      const int acc = tl & 1;
      if (!mbar_wait_warp(smem_u32(&sh->tfull[acc]), (tl >> 1) & 1, status, abort_flag)) break;
      tc_fence_after();
      const int m0 = (t % num_m) * 2 * UBM + static_cast<int>(rank) * UBM;
      const int nt = t / num_m;
      const bool row_ok = m0 + q * 32 + lane < rows;
      // Segments of one 128-byte staging row each: bf16, 64 columns; e4m3, a
      // whole 128-column head of K (e4m3) or half a head of V (64 columns as
      // f16 holding the e4m3-rounded values, the operand the attention's P*V
      // reads without widening).
#pragma unroll 1
      for (int seg = 0; seg < 4; ++seg) {
        const int blk = seg >> 1;
        const int hf = 2 * nt + blk;             // 128-wide block of N
        const bool k_blk = hf < H;
        if (ELT == 1 && k_blk && (seg & 1)) continue;   // e4m3 K head: one segment
        const int col = (ELT == 1 && k_blk) ? blk * 128 : seg * 64;   // within the 256-wide tile
        const int ncols = (ELT == 1 && k_blk) ? 128 : 64;
        uint32_t packed[32];
#pragma unroll
        for (int part = 0; part < 4; ++part) {
          if (part * 32 >= ncols) break;
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + acc * UBN + col + part * 32, r);
          tmem_ld_wait();
          if (ELT == 2) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed[part * 16 + i] = row_ok ? pack_bf16(__uint_as_float(r[2 * i]) * out_scale,
                                                         __uint_as_float(r[2 * i + 1]) * out_scale)
                                             : 0u;
          } else if (k_blk) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t lo = pack_e4m3(__uint_as_float(r[4 * i]) * out_scale,
                                            __uint_as_float(r[4 * i + 1]) * out_scale);
              const uint32_t hi = pack_e4m3(__uint_as_float(r[4 * i + 2]) * out_scale,
                                            __uint_as_float(r[4 * i + 3]) * out_scale);
              packed[part * 8 + i] = row_ok ? (lo | (hi << 16)) : 0u;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed[part * 16 + i] =
                  row_ok ? e4m3x2_to_f16x2(pack_e4m3(__uint_as_float(r[2 * i]) * out_scale,
                                                     __uint_as_float(r[2 * i + 1]) * out_scale))
                         : 0u;
          }
        }
        const bool last = seg == 3 || (ELT == 1 && seg == 2 && 2 * nt + 1 < H);
        if (last) {
          // All of this accumulator has been read: hand it back to the MMA warp.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(tempty0 + acc * 8);
        }
        // Reuse a staging buffer only after its previous TMA store has read it.
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
        uint8_t* sb = stage_buf + buf * UEPI_BYTES;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(sb + lane * 128 + ((c ^ (lane & 7)) * 16)) =
              make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          const CUtensorMap* omap = k_blk ? &k_out_map : &v_out_map;
          tma_store_2d(omap, smem_u32(sb), (hf % H) * 128 + (col % 128), m0 + q * 32);
          bulk_commit();
        }
        buf ^= 1;
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // neither CTA frees TMEM or leaves while the pair still uses it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, U_TMEM_COLS);
  }
}

template <int ELT, bool PAGED>
int pair_gemm_clusters(int device) {
  static std::mutex mu;
  static int cached[64];
  static bool done[64];
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return 0;
  if (!done[device]) {
    cudaFuncSetAttribute(upproj_pair_kernel<ELT, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize, U_SMEM_TOTAL);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(U_THREADS);
    cfg.dynamicSmemBytes = U_SMEM_TOTAL;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, upproj_pair_kernel<ELT, PAGED>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cached[device] = n;
    done[device] = true;
  }
  return cached[device];
}

}  // namespace

cudaError_t launch_upproject(const UpprojArgs& a, cudaStream_t stream) {
  const int elt = a.dtype == MLA_BF16 ? 2 : 1;
  const CUtensorMapDataType dt =
      elt == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint32_t box_k = UBKB / elt;
  const uint64_t HN = static_cast<uint64_t>(a.H) * 128;
  CUtensorMap a_map, wk_map, wuv_map, k_map, v_map;
  const bool paged = a.kv_cache != nullptr;
  PagedA pa = {static_cast<const uint8_t*>(a.kv_cache), paged ? a.cache_rows : nullptr, a.num_cache_rows,
               576 * elt};
  // (paged: a_map is not read; it is encoded over the cache rows to stay valid)
  const bool ok =
      (paged ? encode_2d(&a_map, a.kv_cache, dt, 576, static_cast<uint64_t>(a.num_cache_rows), 576ull * elt,
                         box_k, 1, CU_TENSOR_MAP_SWIZZLE_128B)
             : encode_2d(&a_map, a.c_kv, dt, 512, a.S, 512ull * elt, box_k, UBM, CU_TENSOR_MAP_SWIZZLE_128B)) &&
      encode_2d(&wk_map, a.w_k, dt, 512, HN, 512ull * elt, box_k, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_2d(&wuv_map, a.w_uv, dt, 512, HN, 512ull * elt, box_k, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_2d(&k_map, a.k_nope, dt, HN, a.S, HN * elt, box_k, 32, CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_2d(&v_map, a.v, elt == 2 ? dt : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, HN, a.S, HN * 2, 64, 32,
                      CU_TENSOR_MAP_SWIZZLE_128B);   // V: bf16, or f16 holding e4m3-rounded values
  if (!ok) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int clusters = elt == 2 ? (paged ? pair_gemm_clusters<2, true>(dev) : pair_gemm_clusters<2, false>(dev))
                                : (paged ? pair_gemm_clusters<1, true>(dev) : pair_gemm_clusters<1, false>(dev));
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  // Upper bound on pair tiles (the device reads the chunk's real row count).
  const long long max_tiles = static_cast<long long>((a.S + 2 * UBM - 1) / (2 * UBM)) * a.H;
  const int grid = 2 * static_cast<int>(max_tiles < clusters ? max_tiles : clusters);
  auto kernel = elt == 2 ? (paged ? upproj_pair_kernel<2, true> : upproj_pair_kernel<2, false>)
                         : (paged ? upproj_pair_kernel<1, true> : upproj_pair_kernel<1, false>);
  return launch_pdl(kernel, dim3(grid), dim3(U_THREADS), U_SMEM_TOTAL, stream, a_map, wk_map, wuv_map, k_map, v_map,
                    a.buffer_lengths, a.chunk, int(a.S), a.H, a.out_scale, a.status, pa);
}

}  // namespace mla
