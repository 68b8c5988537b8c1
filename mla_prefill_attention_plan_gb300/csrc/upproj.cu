// Up-projection ("mla_prefill_decode_graph_bf16", Args: w_k, w_uv):
//   K_nope[r, h, :] = s * c_kv[r, :] . w_k[h*128 + :, :]^T
//   V[r, h, :]      = s * c_kv[r, :] . w_uv[h, :, :]^T
// as one GEMM  [rows, 512] x [512, 2*H*128]  whose N axis is the 128-wide
// blocks of w_k (K_nope heads 0..H-1) followed by those of w_uv (V heads).
// Both weights are K-contiguous ([N, K]), exactly the K-major B operand of the
// tensor core; every 128-column block of N is one head of K_nope or of V, so
// the epilogue writes [rows, H, 128] directly.
//
// sm_103a design: persistent CTAs (one per SM) walk 128x256 output tiles.
//   warp 0      TMA producer: A tile 128x(128 B) and two B halves 128x(128 B)
//               per k-block into a 4-stage shared-memory ring (128-byte swizzle)
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma (M=128,
//               N=256, K=16 bf16 / 32 e4m3) from one thread into one of two
//               256-column fp32 accumulators
//   warps 2..5  epilogue: tcgen05.ld a 32-lane quarter of the accumulator,
//               scale, round to the storage type, stage 32x128 B in shared
//               memory and TMA-store it; the second accumulator lets the next
//               tile's MMAs run under this epilogue.
#include <cstdlib>
#include <cstring>

#include "kernels.cuh"

namespace mla {
namespace {

constexpr int BM = 128, BN = 256, BKB = 128;  // tile rows, tile cols, k-block bytes
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BKB;             // 16 KB
constexpr int B_BYTES = BN * BKB;             // 32 KB
constexpr int EPI_BYTES = 32 * 128;           // one 32-row x 128-byte staging buffer
constexpr int SMEM_A = 0;
constexpr int SMEM_B = SMEM_A + STAGES * A_BYTES;
constexpr int SMEM_EPI = SMEM_B + STAGES * B_BYTES;            // 196608
constexpr int SMEM_BAR = SMEM_EPI + 4 * 2 * EPI_BYTES;        // 229376
constexpr int SMEM_TOTAL = SMEM_BAR + 256 + 1024;             // + barriers + alignment slack
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(Smem) <= 256, "barrier block");

template <int ELT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    upproj_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap wk_map,
                  const __grid_constant__ CUtensorMap wuv_map,
                  const __grid_constant__ CUtensorMap k_out_map,
                  const __grid_constant__ CUtensorMap v_out_map, const int32_t* buffer_lengths,
                  int chunk, int S, int H, float out_scale, int32_t* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Smem* sh = reinterpret_cast<Smem*>(smem + SMEM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int rows = buffer_lengths ? buffer_lengths[chunk] : S;
  if (rows <= 0) return;
  if (status && *reinterpret_cast<volatile int32_t*>(status) == MLA_DEV_TIMEOUT) return;
  if (rows > S) rows = S;
  const int num_m = (rows + BM - 1) / BM;
  const int num_n = H;  // 2*H*128 / 256
  const int num_tiles = num_m * num_n;
  constexpr int KB = 512 * ELT / BKB;   // k-blocks: 8 (bf16) or 4 (e4m3)
  constexpr int KSTEP = 32;             // bytes of one MMA's K: 16 bf16 / 32 e4m3
  constexpr uint32_t IDESC = ELT == 2 ? idesc_bf16(BM, BN, false, false) : idesc_e4m3(BM, BN, false, false);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh->tfull[i]), 1);
      mbar_init(smem_u32(&sh->tempty[i]), 4);
    }
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sh->tmem), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem;
  volatile int* abort_flag = &sh->abort;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&a_map);
      prefetch_tmap(&wk_map);
      prefetch_tmap(&wuv_map);
      int stage = 0;
      uint32_t phase = 0;
      int last_ph[STAGES];
      for (int s = 0; s < STAGES; ++s) last_ph[s] = -1;
      for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x) {
        const int m0 = (t % num_m) * BM;
        const int nt = t / num_m;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!(ok = mbar_wait(smem_u32(&sh->empty[stage]), phase ^ 1, status, abort_flag))) break;
          const uint32_t full = smem_u32(&sh->full[stage]);
          mbar_expect_tx(full, A_BYTES + B_BYTES);
          const int x = kb * (BKB / ELT);
          tma_load_2d(smem_u32(smem + SMEM_A + stage * A_BYTES), &a_map, full, x, m0);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int hf = 2 * nt + half;  // 128-wide block of N: K_nope head or V head
            const CUtensorMap* wmap = hf < H ? &wk_map : &wuv_map;
            tma_load_2d(smem_u32(smem + SMEM_B + stage * B_BYTES + half * (B_BYTES / 2)), wmap, full,
                        x, (hf % H) * 128);
          }
          last_ph[stage] = int(phase);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
      // Drain: every issued load lands before the CTA exits.
      volatile int never = 0;
      for (int s = 0; s < STAGES; ++s)
        if (last_ph[s] >= 0) mbar_wait(smem_u32(&sh->full[s]), uint32_t(last_ph[s]), status, &never);
      // ... and every stage release the MMAs committed to this CTA has
      // arrived: an asynchronous arrival must not reach a CTA that has left.
      for (int s = 0; s < STAGES; ++s)
        if (last_ph[s] >= 0) mbar_wait(smem_u32(&sh->empty[s]), uint32_t(last_ph[s]), status, abort_flag);
    }
  } else if (warp == 1) {
    // One elected lane runs the whole loop, waits included; the warp
    // reconverges only at the end (a warp that reconverges while its lane has
    // MMAs in flight stalls until most of them have executed, and the next
    // wait then leaves the tensor pipe idle).
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int tl = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++tl) {
        const int acc = tl & 1;
        if (!(ok = mbar_wait(smem_u32(&sh->tempty[acc]), ((tl >> 1) & 1) ^ 1, status, abort_flag))) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!(ok = mbar_wait(smem_u32(&sh->full[stage]), phase, status, abort_flag))) break;
          tc_fence_after();
          const uint32_t a = smem_u32(smem + SMEM_A + stage * A_BYTES);
          const uint32_t b = smem_u32(smem + SMEM_B + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BKB / KSTEP; ++k) {
            const uint64_t ad = sdesc(a + k * KSTEP, 16, 1024);
            const uint64_t bd = sdesc(b + k * KSTEP, 16, 1024);
            if (ELT == 2) mma_f16_ss(d, ad, bd, IDESC, (kb | k) != 0);
            else mma_f8_ss(d, ad, bd, IDESC, (kb | k) != 0);
          }
          tc_commit(smem_u32(&sh->empty[stage]));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (ok) tc_commit(smem_u32(&sh->tfull[acc]));
      }
      // Drain: every MMA issued so far completes before TMEM is released.
      tc_commit(smem_u32(&sh->drain));
      volatile int never = 0;
      mbar_wait(smem_u32(&sh->drain), 0, status, &never);
    }
    __syncwarp();
  } else {
    // Epilogue warps 2..5: TMEM lane quarter q = warp % 4 holds tile rows 32q..32q+31.
    const int q = warp & 3;
    const uint32_t lane_off = uint32_t(q * 32) << 16;
    uint8_t* stage_buf = smem + SMEM_EPI + (warp - 2) * 2 * EPI_BYTES;
    int buf = 0;
    int tl = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tl) {
      const int acc = tl & 1;
      if (!mbar_wait_warp(smem_u32(&sh->tfull[acc]), (tl >> 1) & 1, status, abort_flag)) break;
      tc_fence_after();
      const int m0 = (t % num_m) * BM;
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
          tmem_ld32(tmem + lane_off + acc * BN + col + part * 32, r);
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
          if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[acc]));
        }
        // Reuse a staging buffer only after its previous TMA store has read it.
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
        uint8_t* sb = stage_buf + buf * EPI_BYTES;
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
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_upproject(const UpprojArgs& a, cudaStream_t stream) {
  const char* pick = std::getenv("MLA_UPPROJ_KERNEL");
  if (!(pick != nullptr && std::strcmp(pick, "single") == 0) && upproject_pair_available(a.dtype))
    return launch_upproject_pair(a, stream);
  const int elt = a.dtype == MLA_BF16 ? 2 : 1;
  const CUtensorMapDataType dt =
      elt == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint32_t box_k = BKB / elt;  // elements in one 128-byte row
  const uint64_t HN = static_cast<uint64_t>(a.H) * 128;
  CUtensorMap a_map, wk_map, wuv_map, k_map, v_map;
  bool ok = encode_2d(&a_map, a.c_kv, dt, 512, a.S, 512ull * elt, box_k, BM, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&wk_map, a.w_k, dt, 512, HN, 512ull * elt, box_k, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&wuv_map, a.w_uv, dt, 512, HN, 512ull * elt, box_k, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&k_map, a.k_nope, dt, HN, a.S, HN * elt, box_k, 32, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&v_map, a.v, elt == 2 ? dt : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, HN, a.S, HN * 2, 64, 32,
                      CU_TENSOR_MAP_SWIZZLE_128B);   // V: bf16, or f16 holding e4m3-rounded values
  if (!ok) return cudaErrorInvalidValue;
  // Upper bound on tiles (the device reads the chunk's real row count).
  const int max_tiles = static_cast<int>((a.S + BM - 1) / BM) * a.H;
  const int grid = max_tiles < sm_count() ? max_tiles : sm_count();
  if (elt == 2) {
    static bool attr2 = false;
    if (!attr2) {
      cudaFuncSetAttribute(upproj_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
      attr2 = true;
    }
    upproj_kernel<2><<<grid, NUM_THREADS, SMEM_TOTAL, stream>>>(a_map, wk_map, wuv_map, k_map, v_map,
                                                              a.buffer_lengths, a.chunk, int(a.S), a.H,
                                                              a.out_scale, a.status);
  } else {
    static bool attr1 = false;
    if (!attr1) {
      cudaFuncSetAttribute(upproj_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
      attr1 = true;
    }
    upproj_kernel<1><<<grid, NUM_THREADS, SMEM_TOTAL, stream>>>(a_map, wk_map, wuv_map, k_map, v_map,
                                                              a.buffer_lengths, a.chunk, int(a.S), a.H,
                                                              a.out_scale, a.status);
  }
  return cudaGetLastError();
}

}  // namespace mla
