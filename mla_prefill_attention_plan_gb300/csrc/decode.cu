// MLA decode in the absorbed form ("mla_prefill_decode_graph_bf16": the graph
// switches to decode by the batch's max sequence length; Args w_uk
// [num_heads, kv_latent_dim, qk_nope_head_dim], w_uv [num_heads, v_head_dim,
// kv_latent_dim], num_partitions_in; the sparse form: d_indices,
// indices_stride, topk_lengths, attn_sink_ptr).
//
// Instead of up-projecting the cache to per-head K and V, the nope part of
// every query head is projected into latent space and attends to the 576-wide
// latent rows straight from the paged cache; the latent result is projected
// back per head.  Four launches:
//
//   1. head_gemm_kernel  q_lat[t, h] = w_uk[h] q_nope[t, h]      (tcgen05 GEMM,
//      M = tokens, N = 512 in four CTAs, K = 128 per head), written with q's rope part as
//      the 576-wide query rows q_full [T*H, 576] bf16.
//   2. decode_attn_kernel  the latent attention over key partitions, on pairs
//      of SMs.  A work item is (sequence, 128 query rows, key partition); the
//      rows are (token, head) pairs of one sequence.  CTA r of the pair owns
//      latent columns [256r, 256r + 256) and rope columns [32r, 32r + 32): it
//      loads only those columns of each 64-key tile, contracts them against
//      the same columns of Q (S_r, M = 128, N = 64, K = 288), sends S_r to
//      the other CTA's shared memory with st.async and adds the S it
//      receives, so both hold the full scores without computing any twice.
//      Both run the same softmax and each accumulates O for its own 256 value
//      columns (P V, N = 256).  The full fp32 O of 128 rows x 512 columns
//      would fill a whole TMEM; split this way each SM holds S (2 x 64
//      columns), O (256) and its half of Q (128), 512 columns in all.
//   3. decode_merge_kernel  merges the partitions' (O, LSE) per row, adds the
//      attention sink to the softmax denominator when given, rounds the latent
//      result to bf16.
//   4. head_gemm_kernel  out[t, h] = w_uv[h] o_lat[t, h]  (N = 128, K = 512).
//
// Key partitions: the context of sequence b (L_b = cached + new tokens, or the
// top-k count in the sparse form) is cut into `parts` ranges of
// ceil(L_b / parts) keys rounded up to the 64-key tile.  The result does not
// depend on where the cuts fall (partials merge exactly by LSE).
#include <algorithm>
#include <mutex>

#include "kernels.cuh"

namespace mla {
namespace {

constexpr float kLn2d = 0.693147180559945309f;
constexpr float kNegInfD = -__builtin_huge_valf();
constexpr float kRescaleLog2 = 8.0f;

// ============================================================ per-head GEMM
// D[r, n] = sum_k A[r, k] B_h[n, k] for head h = blockIdx.y and rows
// [128 blockIdx.x, +128).  A: a 2-D tensor map over bf16 rows, the head's K
// columns starting at column a_col0 + h * a_hstride.  B_h: rows [h N, h N + N)
// of a [H N, K] bf16 tensor map (K contiguous).  fp32 accumulation in TMEM,
// bf16 result at out + row * out_ld + h * out_hstride.  With rope_src set,
// the 64 values at rope_src + row * rope_ld + h * rope_hstride are copied
// after the N results (the query's rope part next to its latent part).
template <int N, int K, int STAGES>
struct HeadGemm {
  static constexpr int KB = K / 64;             // 64-column (128-byte) k-blocks
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BYTES = N * 128;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int SMEM_BAR = STAGES * STAGE;
  static constexpr int SMEM_TOTAL = SMEM_BAR + 256 + 1024;
  static constexpr int NB = N > 256 ? 256 : N;   // N of one MMA (and rows of one B box)
  static constexpr uint32_t TMEM_COLS = N <= 128 ? 128 : (N <= 256 ? 256 : 512);
  static constexpr uint32_t IDESC = idesc_bf16(128, NB, false, false);
  static_assert(K % 64 == 0 && N % NB == 0, "shape");
};

// SPLIT > 1: the head's N * SPLIT output columns are shared by SPLIT CTAs
// (grid.y = H * SPLIT), N each, so that a small M still fills the GPU.
template <int N, int K, int STAGES, int SPLIT>
__global__ void __launch_bounds__(192, 1)
    head_gemm_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap b_map,
                     int a_col0, int a_hstride, __nv_bfloat16* __restrict__ out, long long out_ld,
                     int out_hstride, const __nv_bfloat16* __restrict__ rope_src, long long rope_ld,
                     int rope_hstride, int M, int32_t* status) {
  using C = HeadGemm<N, K, STAGES>;
  struct Bars {
    uint64_t full[STAGES], empty[STAGES], done;
    uint32_t tmem;
    int abort;
  };
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* sh = reinterpret_cast<Bars*>(smem + C::SMEM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y / SPLIT;
  const int nc = blockIdx.y % SPLIT;   // this CTA's N-column block of the head
  const int m0 = blockIdx.x * 128;
  pdl_enter();
  if (timed_out_before(status)) return;   // an earlier kernel timed out: no work

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    mbar_init(smem_u32(&sh->done), 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sh->tmem), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem;
  volatile int* abort_flag = &sh->abort;

  if (warp == 0) {
    if (elect_one()) {
      prefetch_tmap(&a_map);
      prefetch_tmap(&b_map);
      int last[STAGES];
      for (int s = 0; s < STAGES; ++s) last[s] = -1;
      for (int kb = 0; kb < C::KB; ++kb) {
        const int s = kb % STAGES;
        if (kb >= STAGES && !mbar_wait(smem_u32(&sh->empty[s]), ((kb / STAGES) & 1) ^ 1, status, abort_flag))
          break;
        const uint32_t full = smem_u32(&sh->full[s]);
        const uint32_t a = smem_u32(smem + s * C::STAGE);
        mbar_expect_tx(full, C::STAGE);
        tma_load_2d(a, &a_map, full, a_col0 + h * a_hstride + kb * 64, m0);
#pragma unroll
        for (int nb = 0; nb < N; nb += C::NB)
          tma_load_2d(a + C::A_BYTES + nb * 128, &b_map, full, kb * 64, (h * SPLIT + nc) * N + nb);
        last[s] = (kb / STAGES) & 1;
      }
      volatile int never = 0;
      for (int s = 0; s < STAGES; ++s)
        if (last[s] >= 0) mbar_wait(smem_u32(&sh->full[s]), uint32_t(last[s]), status, &never);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (elect_one()) {
      bool ok = true;
      for (int kb = 0; kb < C::KB && ok; ++kb) {
        const int s = kb % STAGES;
        if (!(ok = mbar_wait(smem_u32(&sh->full[s]), (kb / STAGES) & 1, status, abort_flag))) break;
        tc_fence_after();
        const uint32_t a = smem_u32(smem + s * C::STAGE);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = sdesc(a + k * 32, 16, 1024);
#pragma unroll
          for (int nb = 0; nb < N; nb += C::NB)
            mma_f16_ss(tmem + nb, ad, sdesc(a + C::A_BYTES + nb * 128 + k * 32, 16, 1024), C::IDESC,
                       (kb | k) != 0);
        }
        tc_commit(smem_u32(&sh->empty[s]));
      }
      tc_commit(smem_u32(&sh->done));
      volatile int never = 0;
      mbar_wait(smem_u32(&sh->done), 0, status, &never);
    }
    __syncwarp();
  } else {
    // Epilogue: TMEM lane quarter q = warp % 4 holds rows 32q..32q+31.
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    if (mbar_wait_warp(smem_u32(&sh->done), 0, status, abort_flag)) {
      tc_fence_after();
      const bool row_ok = m0 + row < M;
      __nv_bfloat16* dst =
          out + static_cast<long long>(m0 + row) * out_ld + static_cast<long long>(h) * out_hstride + nc * N;
#pragma unroll 1
      for (int c = 0; c < N / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + c * 32, r);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        if (row_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (rope_src != nullptr && row_ok && nc == SPLIT - 1) {
        const uint4* s4 = reinterpret_cast<const uint4*>(rope_src + static_cast<long long>(m0 + row) * rope_ld +
                                                         static_cast<long long>(h) * rope_hstride);
        uint4* d4 = reinterpret_cast<uint4*>(dst + N);
#pragma unroll
        for (int i = 0; i < 8; ++i) d4[i] = s4[i];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ============================================================ latent attention
constexpr int DBN = 64;                           // keys per tile
constexpr int D_KSTAGES = 4;
constexpr int D_KBLK = 64 * 128;                  // 64 keys x 64 latent columns (128 B), 8 KB
constexpr int D_KLAT = 4 * D_KBLK;                // this CTA's 256 latent columns
constexpr int D_KBYTES = D_KLAT + 64 * 64;        // + its 32 rope columns (64 B a key)
constexpr int D_QR_BYTES = 128 * 64;              // Q rope half: 128 rows x 64 B
constexpr int D_X_BYTES = 32 * DBN * 2;           // one warp's partial scores: 32 rows x 64 fp16
constexpr int D_SMEM_K = 0;
constexpr int D_SMEM_QR = D_SMEM_K + D_KSTAGES * D_KBYTES;
constexpr int D_SMEM_XS = D_SMEM_QR + 2 * D_QR_BYTES;        // send buffers [slot][warp]
constexpr int D_SMEM_XR = D_SMEM_XS + 2 * 4 * D_X_BYTES;     // receive buffers [slot][warp]
constexpr int D_SMEM_BAR = D_SMEM_XR + 2 * 4 * D_X_BYTES;
constexpr int D_SMEM_LIST = D_SMEM_BAR + 512;                // this pair's work items
constexpr int kDecodeListMax = 256;                          // items a pair can list
constexpr int kDecodeCompactMax = 32768;                     // item indices worth compacting
constexpr int D_SMEM_TOTAL = D_SMEM_LIST + 4 * kDecodeListMax + 1024;
constexpr int D_THREADS = 320;                    // producer, MMA, 4 softmax warps, 4 exchange warps
constexpr uint32_t D_TMEM_COLS = 512;
constexpr uint32_t D_TM_S = 0, D_TM_O = 128, D_TM_Q = 384;   // S 2 x 64, O 256, Q 128 (bf16 pairs)
constexpr uint32_t IDESC_DS = idesc_bf16(128, DBN, false, false);
constexpr uint32_t IDESC_DPV = idesc_bf16(128, 256, false, true);
static_assert(D_KBYTES % 1024 == 0 && D_SMEM_QR % 1024 == 0 && D_SMEM_XS % 1024 == 0, "alignment");
static_assert(D_SMEM_TOTAL <= 227 * 1024, "shared memory");

struct DecodeSmem {
  uint64_t q_full[2], q_free[2];   // Q rope half in shared memory (TMA), 2 slots
  uint64_t q_ready;                // Q latent half staged in TMEM (4 warps)
  uint64_t k_full[D_KSTAGES], k_empty[D_KSTAGES];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t o_free;                 // 4 warps read O
  uint64_t x_sent[2];              // this CTA's exchange warps have read S of the slot (4 warps)
  uint64_t x_full[2][4];           // the other CTA's partial scores landed (per warp, per slot)
  uint64_t x_empty[2][4];          // the other CTA has read what this CTA sent
  uint64_t drain;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(DecodeSmem) <= 512, "barrier block");

struct DecodeParams {
  const __nv_bfloat16* q_full;     // [R][576]
  const uint32_t* iro;
  const uint32_t* cache_len;
  const int32_t* page_table;
  const int32_t* indices;          // sparse form: [B][indices_stride] physical cache rows, or null
  const int32_t* topk;             // sparse form: [B] valid entries
  __nv_bfloat16* o_part;           // [parts][R][512], each partition's normalised result
  float* lse_part;                 // [parts][R]
  int indices_stride;
  int num_pages, page_size, max_pages;
  int B, H, R, parts, m_tiles;
  int part_keys;                   // > 0: partitions of about this many keys (at most `parts`)
  int dense_tiles;                 // 1: every 64-key tile is 64 consecutive rows of one page
  float scale_log2;
  int32_t* status;
};

// Keys of sequence b: its context (dense) or its top-k list (sparse).
__device__ __forceinline__ long long decode_keys(const DecodeParams& p, int b, long long cb, long long nb) {
  if (p.indices != nullptr) {
    const long long k = p.topk != nullptr ? p.topk[b] : p.indices_stride;
    return max(0ll, min(k, static_cast<long long>(p.indices_stride)));
  }
  return cb + nb;
}
// Partitions of a sequence with L keys: `parts` of them (a count from the
// caller), or, with part_keys set, ceil(L / part_keys) of them capped at
// `parts` (the library's choice: items of about the same size whatever the
// sequence's length).  Each holds ceil(L / count) keys rounded up to the tile.
__device__ __forceinline__ int decode_part_count(const DecodeParams& p, long long L) {
  if (p.part_keys <= 0) return p.parts;
  return static_cast<int>(max(1ll, min(static_cast<long long>(p.parts), (L + p.part_keys - 1) / p.part_keys)));
}
__device__ __forceinline__ long long decode_part_size(long long L, int count) {
  const long long per = (L + count - 1) / count;
  return (per + DBN - 1) / DBN * DBN;
}

struct DItem {
  int b, k;
  int row0;        // first global row of the tile (row = token * H + head)
  int r0;          // first row of the tile within the sequence's rows
  int nrows;       // valid rows
  int qa;          // first token of the sequence
  long long cb;    // cached tokens
  long long L;     // keys of the sequence
  long long key0, key1;   // the partition's keys (key1 before the tile's causal limit)
  int n_kv;        // 64-key tiles to visit
};

__device__ __forceinline__ bool decode_item(const DecodeParams& p, int idx, DItem& it) {
  // Partition-major order: the (sequence, row tile) items of partition 0
  // first, then partition 1, ..., so the items that exist are spread evenly
  // over the SM pairs' static stride; row tiles of one sequence and partition
  // stay adjacent (they read the same keys).
  const int m = idx % p.m_tiles;
  const int kb = idx / p.m_tiles;
  it.b = kb % p.B;
  it.k = kb / p.B;
  it.n_kv = 0;
  const uint32_t qa = p.iro[it.b], qe = p.iro[it.b + 1];
  if (static_cast<long long>(qe) * p.H > p.R) {
    set_status(p.status, MLA_DEV_BAD_OFFSETS);
    return false;
  }
  const long long nb = qe >= qa ? static_cast<long long>(qe - qa) : 0;
  const long long rows_b = nb * p.H;
  it.r0 = m * 128;
  if (it.r0 >= rows_b) return false;
  it.qa = static_cast<int>(qa);
  it.row0 = static_cast<int>(static_cast<long long>(qa) * p.H + it.r0);
  it.nrows = static_cast<int>(min(128ll, rows_b - it.r0));
  it.cb = p.cache_len[it.b];
  it.L = decode_keys(p, it.b, it.cb, nb);
  const int count = decode_part_count(p, it.L);
  if (it.k >= count) return false;
  const long long size = decode_part_size(it.L, count);
  it.key0 = it.k * size;
  it.key1 = min(it.key0 + size, it.L);
  long long hi = it.key1;
  if (p.indices == nullptr) {   // causal: the tile's last token sees keys up to cb + i
    const long long i_last = (it.r0 + it.nrows - 1) / p.H;
    hi = min(hi, it.cb + i_last + 1);
  }
  if (hi <= it.key0) return false;
  it.n_kv = static_cast<int>((hi - it.key0 + DBN - 1) / DBN);
  return true;
}

// The items a pair works on: listed (n >= 0, the pair's share of the items
// that exist, in order), or -- past the list's capacity -- every idx of the
// pair's static stride, the empty ones skipped.
struct DList {
  const int* items;
  int n;
};

__device__ __forceinline__ bool next_decode_item(const DecodeParams& p, int& idx, int stride, int total,
                                                 DItem& it, const DList& wl) {
  if (wl.n >= 0) {
    if (total <= 0) return false;   // a timeout seen at entry: no work
    for (; idx < wl.n; ++idx)
      if (decode_item(p, wl.items[idx], it)) return true;
    return false;
  }
  for (; idx < total; idx += stride)
    if (decode_item(p, idx, it)) return true;
  return false;
}

// Every thread of the CTA: rank the items that exist (idx order) and keep
// those of rank pair_id, pair_id + n_pairs, ... in `mine`, so that the pairs
// get the same number of items whatever the pattern of empty ones (a static
// stride over all indices hands some pairs several times the work of
// others).  Returns the pair's count, or -1 (walk the stride) when the index
// space or the pair's share is too large.  `warp_cnt`: 32 ints of scratch.
__device__ int decode_list(const DecodeParams& p, int total, int pair_id, int n_pairs, int* mine, int* warp_cnt) {
  if (total > kDecodeCompactMax) return -1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nwarps = static_cast<int>(blockDim.x) >> 5;
  int base = 0;
  for (int u0 = 0; u0 < total; u0 += static_cast<int>(blockDim.x)) {
    const int u = u0 + tid;
    DItem t;
    const bool has = u < total && decode_item(p, u, t);
    const uint32_t m = __ballot_sync(0xffffffffu, has);
    if (lane == 0) warp_cnt[warp] = __popc(m);
    __syncthreads();
    int off = base, tot = 0;
    for (int w = 0; w < nwarps; ++w) {
      if (w < warp) off += warp_cnt[w];
      tot += warp_cnt[w];
    }
    if (has) {
      const int r = off + __popc(m & ((1u << lane) - 1u));
      if (r % n_pairs == pair_id && r / n_pairs < kDecodeListMax) mine[r / n_pairs] = u;
    }
    base += tot;
    __syncthreads();   // warp_cnt is rewritten by the next round
  }
  const int n = base > pair_id ? (base - pair_id + n_pairs - 1) / n_pairs : 0;
  return n <= kDecodeListMax ? n : -1;
}

// Physical cache row of key `pos` of sequence b, or -1 (page out of range:
// reported, and the tile reads zeros there).
__device__ __forceinline__ int decode_phys_row(const DecodeParams& p, int b, long long pos) {
  long long row;
  if (p.indices != nullptr) {
    row = p.indices[static_cast<long long>(b) * p.indices_stride + pos];
    if (row < 0 || row >= static_cast<long long>(p.num_pages) * p.page_size) {
      set_status(p.status, MLA_DEV_BAD_PAGE);
      return -1;
    }
    return static_cast<int>(row);
  }
  const long long pi = pos / p.page_size;
  const int page = pi < p.max_pages ? p.page_table[static_cast<long long>(b) * p.max_pages + pi] : -1;
  if (page < 0 || page >= p.num_pages) {
    set_status(p.status, MLA_DEV_BAD_PAGE);
    return -1;
  }
  return static_cast<int>(static_cast<long long>(page) * p.page_size + pos % p.page_size);
}

// 64 key rows of a stage from the cache, 16 bytes per cp.async: lane l holds
// the cache rows of keys l (ra) and l + 32 (rb); each warp instruction copies
// 32 / CH whole rows (CH = 16-byte chunks a row), chunk l % CH of row
// RPI * i + l / CH, into the swizzled layout a tensor-map tile load would give
// (SW128 for 128-byte rows, SW64 for 64-byte rows).  `col0` points at the
// columns to copy in cache row 0.
template <int ROW_BYTES>
__device__ __forceinline__ void key_rows_cp_async(uint32_t dst, const uint8_t* col0, int ra, int rb) {
  constexpr int CH = ROW_BYTES / 16;
  constexpr int RPI = 32 / CH;
  constexpr int ITERS = 64 / RPI;
  const int lane = threadIdx.x & 31;
  const int c = lane % CH;
  const uint8_t* src = col0 + c * 16;
#pragma unroll
  for (int i = 0; i < ITERS; ++i) {
    const int r = RPI * i + lane / CH;
    const int row = __shfl_sync(0xffffffffu, i < ITERS / 2 ? ra : rb, r & 31);
    const int sw = ROW_BYTES == 128 ? (r & 7) : ((r >> 1) & 3);
    cp_async16(dst + r * ROW_BYTES + ((c ^ sw) << 4), src + static_cast<size_t>(row) * 1152);
  }
}

// A stage's cp.async rows have landed (all but the newest N groups of the
// warp): fence them into the async proxy the MMAs read through, then arrive
// on the stage's barrier.
template <int N>
__device__ __forceinline__ void key_rows_landed(uint32_t bar) {
  cp_async_wait<N>();
  fence_async_smem();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// DENSE: every 64-key tile is 64 consecutive rows of one page, loaded as
// rectangular tiles; otherwise (page size not a multiple of 64, or sparse
// lists) the rows are copied one by one with cp.async.  Two instantiations,
// so that the dense one carries no trace of the other path.
template <bool DENSE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(D_THREADS, 1)
    decode_attn_kernel(const __grid_constant__ CUtensorMap qr_map, const __grid_constant__ CUtensorMap kl_map,
                       const __grid_constant__ CUtensorMap kr_map, const __grid_constant__ CUtensorMap kl1_map,
                       const __grid_constant__ CUtensorMap kr1_map, const DecodeParams p, int total_items,
                       const uint8_t* __restrict__ cache_rows) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DecodeSmem* sh = reinterpret_cast<DecodeSmem*>(smem + D_SMEM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t other = rank ^ 1u;
  const int pair_id = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;
  int32_t* status = p.status;
  pdl_enter();

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh->q_full[i]), 1);
      mbar_init(smem_u32(&sh->q_free[i]), 1);
      mbar_init(smem_u32(&sh->s_full[i]), 1);
      mbar_init(smem_u32(&sh->p_full[i]), 4);
      mbar_init(smem_u32(&sh->o_done[i]), 1);
      mbar_init(smem_u32(&sh->x_sent[i]), 4);
      for (int w = 0; w < 4; ++w) {
        mbar_init(smem_u32(&sh->x_full[i][w]), 1);
        mbar_init(smem_u32(&sh->x_empty[i][w]), 1);
      }
    }
    mbar_init(smem_u32(&sh->q_ready), 4);
    for (int s = 0; s < D_KSTAGES; ++s) {
      mbar_init(smem_u32(&sh->k_full[s]), 1);
      mbar_init(smem_u32(&sh->k_empty[s]), 1);
    }
    mbar_init(smem_u32(&sh->o_free), 4);
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort = timed_out_before(status) ? 1 : 0;
    fence_mbar_init();
    // The first phase of every receive slot expects one warp's scores.
    for (int i = 0; i < 2; ++i)
      for (int w = 0; w < 4; ++w) mbar_expect_tx(smem_u32(&sh->x_full[i][w]), D_X_BYTES);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sh->tmem), D_TMEM_COLS);
    tmem_relinquish();
  }
  // The pair's work list (both CTAs compute the same one); the send buffers,
  // unused until the first exchange, hold the scan's scratch.
  const DList wl{reinterpret_cast<const int*>(smem + D_SMEM_LIST),
                 decode_list(p, total_items, pair_id, n_pairs, reinterpret_cast<int*>(smem + D_SMEM_LIST),
                             reinterpret_cast<int*>(smem + D_SMEM_XS))};
  const int istart = wl.n >= 0 ? 0 : pair_id;
  const int istep = wl.n >= 0 ? 1 : n_pairs;
  tc_fence_before();
  cluster_sync();   // barriers of both CTAs initialised (the other CTA stores into them)
  tc_fence_after();
  const int total = cluster_any(&sh->abort) ? 0 : total_items;
  const uint32_t tmem = sh->tmem;
  volatile int* abort_flag = &sh->abort;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      prefetch_tmap(&qr_map);
      prefetch_tmap(DENSE ? &kl_map : &kl1_map);
      prefetch_tmap(DENSE ? &kr_map : &kr1_map);
    }
    __syncwarp();
    uint32_t g = 0, it_n = 0;
    uint32_t q_issued = 0, k_issued = 0;   // Q-rope and K-tile loads issued
    int k_pend = -1;                       // stage whose cp.async rows are in flight
    bool ok = true;
    DItem it;
    const int lat_x = 256 * static_cast<int>(rank);
    const int rope_x = 512 + 32 * static_cast<int>(rank);
    for (int idx = istart; ok && next_decode_item(p, idx, istep, total, it, wl); idx += istep) {
      const int qs = it_n & 1;
      if (it_n >= 2 &&
          !(ok = mbar_wait_warp(smem_u32(&sh->q_free[qs]), ((it_n >> 1) & 1) ^ 1, status, abort_flag)))
        break;
      if (elect_one()) {
        const uint32_t qf = smem_u32(&sh->q_full[qs]);
        mbar_expect_tx(qf, D_QR_BYTES);
        tma_load_2d(smem_u32(smem + D_SMEM_QR + qs * D_QR_BYTES), &qr_map, qf, rope_x, it.row0);
      }
      __syncwarp();
      ++q_issued;
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t gj = g + j;
        const int st = gj % D_KSTAGES;
        const long long pos0 = it.key0 + static_cast<long long>(j) * DBN;
        // The tile's cache rows (a page-table or index read) before waiting for
        // its stage, so that the read's latency overlaps the wait.
        int ra, rb;
        if constexpr (DENSE) {
          // 64 consecutive positions, all in one page.
          ra = decode_phys_row(p, it.b, pos0);
          if (ra < 0) ra = p.num_pages * p.page_size;   // past the end: reads zeros
          rb = 0;
        } else {
          const long long pa = pos0 + lane, pb = pos0 + 32 + lane;
          ra = pa < it.L ? decode_phys_row(p, it.b, pa) : 0;
          rb = pb < it.L ? decode_phys_row(p, it.b, pb) : 0;
          if (ra < 0) ra = 0;   // reported; the scores of such a key are wrong, the status says so
          if (rb < 0) rb = 0;
        }
        if (gj >= D_KSTAGES &&
            !(ok = mbar_wait_warp(smem_u32(&sh->k_empty[st]), ((gj / D_KSTAGES) & 1) ^ 1, status, abort_flag)))
          break;
        const uint32_t kf = smem_u32(&sh->k_full[st]);
        const uint32_t kd = smem_u32(smem + D_SMEM_K + st * D_KBYTES);
        if constexpr (DENSE) {
          if (elect_one()) {
            mbar_expect_tx(kf, D_KBYTES);
#pragma unroll
            for (int c = 0; c < 4; ++c) tma_load_2d(kd + c * D_KBLK, &kl_map, kf, lat_x + 64 * c, ra);
            tma_load_2d(kd + D_KLAT, &kr_map, kf, rope_x, ra);
          }
        } else {
          // Any rows, 16 bytes per cp.async (one-row TMA gathers cost far
          // more per byte); the previous stage is counted once its rows land.
          const uint8_t* cache = cache_rows;
#pragma unroll
          for (int c = 0; c < 4; ++c) key_rows_cp_async<128>(kd + c * D_KBLK, cache + (lat_x + 64 * c) * 2, ra, rb);
          key_rows_cp_async<64>(kd + D_KLAT, cache + rope_x * 2, ra, rb);
          cp_async_commit();
          if (k_pend >= 0) key_rows_landed<1>(smem_u32(&sh->k_full[k_pend]));
          k_pend = st;
        }
        __syncwarp();
        ++k_issued;
      }
      if constexpr (!DENSE) {   // the item's last stage, before any other wait
        if (k_pend >= 0) key_rows_landed<0>(smem_u32(&sh->k_full[k_pend]));
        k_pend = -1;
      }
      g += it.n_kv;
      ++it_n;
    }
    if constexpr (!DENSE) {
      if (k_pend >= 0) key_rows_landed<0>(smem_u32(&sh->k_full[k_pend]));
    }
    // Every issued load lands before the CTA leaves: the last phase of each
    // slot and stage that a load used.
    volatile int never = 0;
    for (uint32_t s = 0; s < 2; ++s)
      if (q_issued > s) {
        const uint32_t last = s + 2 * ((q_issued - 1 - s) / 2);
        mbar_wait_warp(smem_u32(&sh->q_full[s]), (last >> 1) & 1, status, &never);
      }
    for (uint32_t s = 0; s < D_KSTAGES; ++s)
      if (k_issued > s) {
        const uint32_t last = s + D_KSTAGES * ((k_issued - 1 - s) / D_KSTAGES);
        mbar_wait_warp(smem_u32(&sh->k_full[s]), (last / D_KSTAGES) & 1, status, &never);
      }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      uint32_t g = 0, it_n = 0;
      DItem it;
      bool ok = true;
      for (int idx = istart; ok && next_decode_item(p, idx, istep, total, it, wl); idx += istep) {
        const int qs = it_n & 1;
        if (!(ok = mbar_wait(smem_u32(&sh->q_ready), it_n & 1, status, abort_flag))) break;
        if (!(ok = mbar_wait(smem_u32(&sh->q_full[qs]), (it_n >> 1) & 1, status, abort_flag))) break;
        const uint32_t qr = smem_u32(smem + D_SMEM_QR + qs * D_QR_BYTES);
        const int n = it.n_kv;
        auto issue_s = [&](int j) -> bool {
          const uint32_t gj = g + j;
          const int st = gj % D_KSTAGES;
          if (!mbar_wait(smem_u32(&sh->k_full[st]), (gj / D_KSTAGES) & 1, status, abort_flag)) return false;
          // The exchange warps have read S of the tile two back from this buffer.
          if (gj >= 2 && !mbar_wait(smem_u32(&sh->x_sent[gj & 1]), ((gj >> 1) - 1) & 1, status, abort_flag))
            return false;
          tc_fence_after();
          const uint32_t kd = smem_u32(smem + D_SMEM_K + st * D_KBYTES);
          const uint32_t d = tmem + D_TM_S + (gj & 1) * DBN;
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)   // latent: A = Q half in TMEM, 16 bf16 = 8 columns a step
            mma_f16_ts(d, tmem + D_TM_Q + kk * 8, sdesc(kd + (kk >> 2) * D_KBLK + (kk & 3) * 32, 16, 1024),
                       IDESC_DS, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)    // rope: both operands in shared memory, 64-byte rows
            mma_f16_ss(d, sdesc(qr + kk * 32, 16, 512, kSwizzle64),
                       sdesc(kd + D_KLAT + kk * 32, 16, 512, kSwizzle64), IDESC_DS, 1);
          tc_commit(smem_u32(&sh->s_full[gj & 1]));
          if (j == n - 1) tc_commit(smem_u32(&sh->q_free[qs]));
          return true;
        };
        auto issue_pv = [&](int j) -> bool {
          const uint32_t gj = g + j;
          const int st = gj % D_KSTAGES;
          if (!mbar_wait(smem_u32(&sh->p_full[gj & 1]), (gj >> 1) & 1, status, abort_flag)) return false;
          if (j == 0 && it_n >= 1 && !mbar_wait(smem_u32(&sh->o_free), (it_n - 1) & 1, status, abort_flag))
            return false;
          tc_fence_after();
          const uint32_t kd = smem_u32(smem + D_SMEM_K + st * D_KBYTES);
          const uint32_t pa = tmem + D_TM_S + (gj & 1) * DBN;
#pragma unroll
          for (int kk = 0; kk < DBN / 16; ++kk)   // V = the latent columns, MN-major (64-column blocks)
            mma_f16_ts(tmem + D_TM_O, pa + kk * 8, sdesc(kd + kk * 2048, D_KBLK, 1024), IDESC_DPV,
                       (j > 0 || kk > 0));
          tc_commit(smem_u32(&sh->o_done[gj & 1]));
          tc_commit(smem_u32(&sh->k_empty[st]));
          return true;
        };
        ok = issue_s(0);
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
  } else if (warp >= 6) {
    // ------------------------------------------------------------ exchange
    // Every tile's partial scores of this warp's 32 rows, read from TMEM as
    // soon as the S MMA completes, rounded to fp16 and shipped to the other
    // CTA's receive slot gj & 1 with one bulk copy, once it has read what this
    // warp sent there two tiles ago.  (Both CTAs add the same two rounded
    // halves, so both get the same scores.)
    const int q4 = warp & 3;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    constexpr uint32_t kSlotStep = 4 * D_X_BYTES;
    constexpr uint32_t kBarSlot = 4 * 8;
    const uint32_t xs_mine = smem_u32(smem + D_SMEM_XS + q4 * D_X_BYTES);
    const uint32_t xr_other = cluster_addr(smem_u32(smem + D_SMEM_XR + q4 * D_X_BYTES), other);
    const uint32_t xf_other = cluster_addr(smem_u32(&sh->x_full[0][q4]), other);
    uint32_t g = 0;
    bool ok = true;
    DItem it;
    for (int idx = istart; ok && next_decode_item(p, idx, istep, total, it, wl); idx += istep) {
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t gj = g + j;
        const uint32_t sb = gj & 1, use = gj >> 1;
        if (!(ok = mbar_wait_warp(smem_u32(&sh->s_full[sb]), use & 1, status, abort_flag))) break;
        tc_fence_after();
        uint32_t x[DBN];
        tmem_ld32(tmem + lane_off + D_TM_S + sb * DBN, *reinterpret_cast<uint32_t(*)[32]>(x));
        tmem_ld32(tmem + lane_off + D_TM_S + sb * DBN + 32, *reinterpret_cast<uint32_t(*)[32]>(x + 32));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh->x_sent[sb]));
        uint32_t h[DBN / 2];
#pragma unroll
        for (int k = 0; k < DBN / 2; ++k) h[k] = pack_f16(__uint_as_float(x[2 * k]), __uint_as_float(x[2 * k + 1]));
        if (use > 0 && !(ok = mbar_wait_warp(smem_u32(&sh->x_empty[sb][q4]), (use - 1) & 1, status, abort_flag)))
          break;
        uint8_t* sbuf = smem + D_SMEM_XS + sb * kSlotStep + q4 * D_X_BYTES;
#pragma unroll
        for (int c = 0; c < DBN / 8; ++c)
          *reinterpret_cast<uint4*>(sbuf + c * 512 + lane * 16) = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0)
          bulk_copy_to_cluster(xr_other + sb * kSlotStep, xs_mine + sb * kSlotStep, D_X_BYTES,
                               xf_other + sb * kBarSlot);
      }
      g += it.n_kv;
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    const float sl2 = p.scale_log2;
    const float2 sl2v = make_float2(sl2, sl2);
    constexpr uint32_t kSlotStep = 4 * D_X_BYTES;
    constexpr uint32_t kBarSlot = 4 * 8;
    const uint32_t xe_other = cluster_addr(smem_u32(&sh->x_empty[0][q4]), other);
    uint32_t g = 0, it_n = 0;
    uint32_t taken0 = 0, taken1 = 0;   // phases of each receive slot this warp has consumed
    bool ok = true;

    // The item's Q latent half (256 bf16 of the row) into TMEM columns
    // D_TM_Q..+127; the MMAs read it from there.
    auto stage_q = [&](const DItem& n_it) {
      uint32_t v[128];
      if (row < n_it.nrows) {
        const uint4* src = reinterpret_cast<const uint4*>(p.q_full + static_cast<long long>(n_it.row0 + row) * 576 +
                                                          256 * rank);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint4 x = src[i];
          v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 128; ++i) v[i] = 0u;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_st32(tmem + lane_off + D_TM_Q + c * 32, v + c * 32);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->q_ready));
    };

    int idx = istart;
    DItem it;
    bool have = next_decode_item(p, idx, istep, total, it, wl);
    if (have) stage_q(it);
    while (have && ok) {
      // This row's keys: [key0, hi) of the partition, causal for dense decode.
      const long long tok = (it.r0 + row) / p.H;
      long long hi = it.key1;
      if (p.indices == nullptr) hi = min(hi, it.cb + tok + 1);
      if (row >= it.nrows) hi = it.key0;
      float m_run = kNegInfD, l_run = 0.f;
      for (int j = 0; j < it.n_kv && ok; ++j) {
        const uint32_t gj = g + j;
        const uint32_t sb = gj & 1;
        // This CTA's partial scores of the tile (rounded to fp16 as the
        // exchange warp sends them), then the other CTA's.
        if (!(ok = mbar_wait_warp(smem_u32(&sh->s_full[sb]), (gj >> 1) & 1, status, abort_flag))) break;
        tc_fence_after();
        uint32_t own[DBN];
        tmem_ld32(tmem + lane_off + D_TM_S + sb * DBN, *reinterpret_cast<uint32_t(*)[32]>(own));
        tmem_ld32(tmem + lane_off + D_TM_S + sb * DBN + 32, *reinterpret_cast<uint32_t(*)[32]>(own + 32));
        const uint32_t taken = sb ? taken1 : taken0;
        if (!(ok = mbar_wait_warp(smem_u32(&sh->x_full[sb][q4]), taken & 1, status, abort_flag))) break;
        if (sb) ++taken1; else ++taken0;
        uint32_t theirs[DBN / 2];
        const uint8_t* rbuf = smem + D_SMEM_XR + sb * kSlotStep + q4 * D_X_BYTES;
#pragma unroll
        for (int c = 0; c < DBN / 8; ++c) {
          const uint4 y = *reinterpret_cast<const uint4*>(rbuf + c * 512 + lane * 16);
          theirs[4 * c] = y.x; theirs[4 * c + 1] = y.y; theirs[4 * c + 2] = y.z; theirs[4 * c + 3] = y.w;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_expect_tx(smem_u32(&sh->x_full[sb][q4]), D_X_BYTES);   // the slot's next phase
          mbar_arrive_cluster(xe_other + sb * kBarSlot);              // the other CTA may send again
        }
        tmem_ld_wait();
        float x[DBN];
#pragma unroll
        for (int k = 0; k < DBN / 2; ++k) {
          const float2 a = f16x2_to_float2(pack_f16(__uint_as_float(own[2 * k]), __uint_as_float(own[2 * k + 1])));
          const float2 b = f16x2_to_float2(theirs[k]);
          x[2 * k] = a.x + b.x;
          x[2 * k + 1] = a.y + b.y;
        }
        // Mask keys outside [key0, hi) of this row.
        const long long lim = hi - (it.key0 + static_cast<long long>(j) * DBN);
        if (lim < DBN) {
#pragma unroll
          for (int k = 0; k < DBN; ++k) x[k] = k < lim ? x[k] : kNegInfD;
        }
        float mx = fmax3(x[0], x[1], x[2]);
#pragma unroll
        for (int k = 3; k < DBN - 1; k += 2) mx = fmax3(mx, x[k], x[k + 1]);
        mx = fmaxf(mx, x[DBN - 1]);
        const float m_new = fmaxf(m_run, mx * sl2);
        const bool need = m_new > m_run + kRescaleLog2;
        const float f = need ? ex2(m_run - m_new) : 1.0f;
        if (need) m_run = m_new;
        const float msub = m_run == kNegInfD ? 0.f : m_run;
        const float2 negm = make_float2(-msub, -msub);
        uint32_t pk[DBN / 2];
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int k = 0; k < DBN / 2; ++k) {
          const float2 t = __ffma2_rn(make_float2(x[2 * k], x[2 * k + 1]), sl2v, negm);
          const float2 e = make_float2(ex2(t.x), ex2(t.y));
          acc[k & 1] = __fadd2_rn(acc[k & 1], e);
          pk[k] = pack_bf16(e.x, e.y);
        }
        const float2 a = __fadd2_rn(acc[0], acc[1]);
        l_run = l_run * f + (a.x + a.y);
        if (j == it.n_kv - 1 && it.key0 + static_cast<long long>(j + 1) * DBN > it.key1) {
          // Keys past the partition in the last tile: zero this CTA's latent
          // columns of those rows (stale or non-finite cache slots) before P V.
          const long long vlim = it.key1 - (it.key0 + static_cast<long long>(j) * DBN);
          const int st = gj % D_KSTAGES;
          const int vr = row >> 1, half = row & 1;
          if (vr >= vlim) {
            uint8_t* base = smem + D_SMEM_K + st * D_KBYTES + vr * 128;
#pragma unroll
            for (int c = 2 * half; c < 2 * half + 2; ++c)
#pragma unroll
              for (int i = 0; i < 8; ++i) reinterpret_cast<uint4*>(base + c * D_KBLK)[i] = make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
        }
        tmem_st32(tmem + lane_off + D_TM_S + sb * DBN, pk);
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // Rescale O only when the row maximum grew by more than 2^8, once
          // P V of the previous tile has completed.
          if (!(ok = mbar_wait_warp(smem_u32(&sh->o_done[(gj - 1) & 1]), ((gj - 1) >> 1) & 1, status, abort_flag)))
            break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t r[32];
            const uint32_t ta = tmem + lane_off + D_TM_O + c * 32;
            tmem_ld32(ta, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
            tmem_st32(ta, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh->p_full[sb]));
      }
      if (!ok) break;
      g += it.n_kv;
      int nidx = idx + istep;
      DItem nx;
      const bool have_next = next_decode_item(p, nidx, istep, total, nx, wl);
      // Every S MMA of this item has completed (its last s_full): the next
      // item's Q may replace this one's in TMEM.
      if (have_next) stage_q(nx);
      // ---------------------------------------------------------- epilogue
      if (!(ok = mbar_wait_warp(smem_u32(&sh->o_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, status, abort_flag)))
        break;
      tc_fence_after();
      const bool store = row < it.nrows;
      const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
      const long long grow = it.row0 + row;
      __nv_bfloat16* dst = p.o_part + (static_cast<long long>(it.k) * p.R + grow) * 512 + 256 * rank;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + D_TM_O + c * 32, r);
        tmem_ld_wait();
        if (store) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            d4[i] = make_uint4(pack_bf16(__uint_as_float(r[8 * i]) * inv, __uint_as_float(r[8 * i + 1]) * inv),
                               pack_bf16(__uint_as_float(r[8 * i + 2]) * inv, __uint_as_float(r[8 * i + 3]) * inv),
                               pack_bf16(__uint_as_float(r[8 * i + 4]) * inv, __uint_as_float(r[8 * i + 5]) * inv),
                               pack_bf16(__uint_as_float(r[8 * i + 6]) * inv, __uint_as_float(r[8 * i + 7]) * inv));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->o_free));
      if (store && rank == 0)
        p.lse_part[static_cast<long long>(it.k) * p.R + grow] =
            l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2d : kNegInfD;
      it = nx;
      idx = nidx;
      have = have_next;
      ++it_n;
    }
    if (!ok) {
      // Aborted: the other CTA may still be copying into a slot this warp
      // handed back; let those copies land (briefly) before the CTA leaves.
      volatile int never = 0;
      mbar_wait_warp(smem_u32(&sh->x_full[0][q4]), taken0 & 1, status, &never, 10000000ull);
      mbar_wait_warp(smem_u32(&sh->x_full[1][q4]), taken1 & 1, status, &never, 10000000ull);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // neither CTA leaves while the other may still store into it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, D_TMEM_COLS);
  }
}

// ============================================================ partition merge
// One row (token, head) per 64 threads, 8 latent columns (one 16-byte load) a
// thread: merge the partitions' (O, LSE) by LSE, add the attention sink (a
// logit with no value) to the denominator when given, and round the latent
// result to bf16.  Each CTA merges a contiguous range of rows, four at a time.
// The sequence of a row is found once and then followed as the token
// advances; four partitions' partial rows are requested before any is used,
// and the grid is one wave of four CTAs per SM.
__global__ void __launch_bounds__(256, 4) decode_merge_kernel(const DecodeParams p, __nv_bfloat16* __restrict__ o_lat,
                                                           float* __restrict__ lse_out,
                                                           const float* __restrict__ sink) {
  pdl_enter();
  if (timed_out_before(p.status)) return;
  constexpr int KU = 4;                        // partitions loaded together
  constexpr int RPP = 4;                       // rows per pass of the CTA (64 threads a row)
  const int sub = threadIdx.x >> 6;            // row within the CTA's group of rows
  const int c = (threadIdx.x & 63) * 8;        // first latent column (16 bytes of bf16)
  const long long per = ((p.R + gridDim.x - 1) / gridDim.x + RPP - 1) / RPP * RPP;
  const long long r_begin = static_cast<long long>(blockIdx.x) * per;
  const long long r_end = min(static_cast<long long>(p.R), r_begin + per);
  int b = -1;
  uint32_t qa = 0, qe = 0;
  for (long long grow = r_begin + sub; grow < r_end; grow += RPP) {
    const int t = static_cast<int>(grow / p.H);
    if (b < 0 || static_cast<uint32_t>(t) >= qe || static_cast<uint32_t>(t) < qa) {
      int lo = 0, hi_b = p.B;                  // largest b with iro[b] <= t
      while (hi_b - lo > 1) {
        const int mid = (lo + hi_b) >> 1;
        if (__ldg(p.iro + mid) <= static_cast<uint32_t>(t)) lo = mid; else hi_b = mid;
      }
      b = lo;
      qa = __ldg(p.iro + b);
      qe = __ldg(p.iro + b + 1);
    }
    if (!(qa <= static_cast<uint32_t>(t) && static_cast<uint32_t>(t) < qe)) {
      // A token outside every sequence: zeros, so the projection reads no garbage.
      *reinterpret_cast<uint4*>(o_lat + grow * 512 + c) = make_uint4(0u, 0u, 0u, 0u);
      if (lse_out != nullptr && c == 0) lse_out[grow] = kNegInfD;
      b = -1;
      continue;
    }
    const long long cb = __ldg(p.cache_len + b);
    const long long L = decode_keys(p, b, cb, static_cast<long long>(qe - qa));
    long long lim = L;
    if (p.indices == nullptr) lim = min(lim, cb + (t - static_cast<long long>(qa)) + 1);
    const int count = decode_part_count(p, L);
    const long long size = decode_part_size(L, count);
    // Partitions holding keys the row sees: 0 .. used - 1.
    const int used = static_cast<int>(min(static_cast<long long>(count), (lim + size - 1) / size));
    // One pass: each group of KU partitions is loaded whole, then merged into
    // the running (max, sum, O) by LSE.
    float mx = kNegInfD;
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float tot = 0.f;
    for (int k0 = 0; k0 < used; k0 += KU) {
      uint4 raw[KU];
      float lk[KU];
#pragma unroll
      for (int i = 0; i < KU; ++i) {
        const int k = k0 + i;
        const long long at = static_cast<long long>(k) * p.R + grow;
        lk[i] = k < used ? __ldg(p.lse_part + at) : kNegInfD;
        raw[i] = k < used ? __ldg(reinterpret_cast<const uint4*>(p.o_part + at * 512 + c))
                          : make_uint4(0u, 0u, 0u, 0u);
      }
      float cm = lk[0];
#pragma unroll
      for (int i = 1; i < KU; ++i) cm = fmaxf(cm, lk[i]);
      const float nm = fmaxf(mx, cm);
      if (nm == kNegInfD) continue;
      const float r = mx == kNegInfD ? 0.f : __expf(mx - nm);
      tot *= r;
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] *= r;
#pragma unroll
      for (int i = 0; i < KU; ++i) {
        const float w = lk[i] == kNegInfD ? 0.f : __expf(lk[i] - nm);
        tot += w;
        const uint32_t u[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          o[2 * j] += w * bf16_lo(u[j]);
          o[2 * j + 1] += w * bf16_hi(u[j]);
        }
      }
      mx = nm;
    }
    float lse = tot > 0.f ? mx + __logf(tot) : kNegInfD;
    float w = tot > 0.f ? 1.0f / tot : 0.f;
    if (sink != nullptr) {
      // The sink joins the softmax denominator: LSE' = log(e^LSE + e^sink).
      const float s = sink[b];
      const float m2 = fmaxf(lse, s);
      const float e1 = lse == kNegInfD ? 0.f : __expf(lse - m2), e2 = __expf(s - m2);
      const float lse2 = m2 + __logf(e1 + e2);
      w *= lse == kNegInfD ? 0.f : __expf(lse - lse2);
      lse = lse2;
    }
    *reinterpret_cast<uint4*>(o_lat + grow * 512 + c) =
        make_uint4(pack_bf16(o[0] * w, o[1] * w), pack_bf16(o[2] * w, o[3] * w), pack_bf16(o[4] * w, o[5] * w),
                   pack_bf16(o[6] * w, o[7] * w));
    if (lse_out != nullptr && c == 0) lse_out[grow] = lse;
  }
}

// Two-CTA clusters of the attention kernel the current device can keep
// resident, or 0.
template <bool DENSE>
int decode_clusters(int device) {
  static std::mutex mu;
  static int cached[64];
  static bool done[64];
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return 0;
  if (!done[device]) {
    cudaFuncSetAttribute(decode_attn_kernel<DENSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, D_SMEM_TOTAL);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(D_THREADS);
    cfg.dynamicSmemBytes = D_SMEM_TOTAL;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_attn_kernel<DENSE>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cached[device] = n;
    done[device] = true;
  }
  return cached[device];
}

template <int N, int K, int STAGES, int SPLIT = 1>
cudaError_t launch_head_gemm(const CUtensorMap& a_map, const CUtensorMap& b_map, int a_col0, int a_hstride,
                             __nv_bfloat16* out, long long out_ld, int out_hstride, const __nv_bfloat16* rope_src,
                             long long rope_ld, int rope_hstride, int M, int H, int32_t* status,
                             cudaStream_t stream) {
  using C = HeadGemm<N, K, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(head_gemm_kernel<N, K, STAGES, SPLIT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_TOTAL);
  if (e != cudaSuccess) return e;
  const dim3 grid((M + 127) / 128, H * SPLIT);
  return launch_pdl(head_gemm_kernel<N, K, STAGES, SPLIT>, grid, dim3(192), C::SMEM_TOTAL, stream, a_map, b_map,
                    a_col0, a_hstride, out, out_ld, out_hstride, rope_src, rope_ld, rope_hstride, M, status);
}

}  // namespace

DecodeLayout decode_layout(int T, int H, int parts) {
  const size_t R = static_cast<size_t>(T) * H;
  DecodeLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = (off + bytes + 255) / 256 * 256;
    return at;
  };
  L.q_full = take(R * 576 * 2);
  L.o_part = take(static_cast<size_t>(parts) * R * 512 * 2);
  L.lse_part = take(static_cast<size_t>(parts) * R * 4);
  L.o_lat = take(R * 512 * 2);
  L.total = off;
  return L;
}

DecodePartitioning decode_partitioning(int B, int H, int max_new, int max_keys) {
  // Items of about the same size, about one per SM pair (each pair gets an
  // equal share of the items, so more items buy no balance, only more partial
  // results to merge: two per pair measured 3 % slower on the top-2048 sparse
  // decode), each between 256 and 2048 keys; at most kDecodeMaxParts a
  // sequence.
  const long long pairs = std::max(1, sm_count() / 2);
  const long long m_tiles = (static_cast<long long>(std::max(1, max_new)) * H + 127) / 128;
  const long long keys = std::max(1, max_keys);
  long long pk = static_cast<long long>(B) * m_tiles * keys / pairs;
  pk = std::min<long long>(2048, std::max<long long>(256, (pk + 63) / 64 * 64));
  DecodePartitioning d;
  d.part_keys = static_cast<int>(pk);
  d.parts = static_cast<int>(std::min<long long>(kDecodeMaxParts, std::max(1ll, (keys + pk - 1) / pk)));
  return d;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const int H = a.H, T = a.T;
  const long long R = static_cast<long long>(T) * H;
  if (T == 0) return cudaSuccess;
  const DecodeLayout L = decode_layout(T, H, a.parts);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  __nv_bfloat16* q_full = reinterpret_cast<__nv_bfloat16*>(ws + L.q_full);
  __nv_bfloat16* o_part = reinterpret_cast<__nv_bfloat16*>(ws + L.o_part);
  float* lse_part = reinterpret_cast<float*>(ws + L.lse_part);
  __nv_bfloat16* o_lat = reinterpret_cast<__nv_bfloat16*>(ws + L.o_lat);
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

  // 1. q_lat = w_uk[h] q_nope, with the rope part alongside: q_full [T*H, 576].
  CUtensorMap qa_map, wuk_map;
  if (!encode_2d(&qa_map, a.q, bf, static_cast<uint64_t>(H) * 192, T, static_cast<uint64_t>(H) * 384, 64, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&wuk_map, a.w_uk, bf, 128, static_cast<uint64_t>(H) * 512, 256, 64, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // Four CTAs a head, 128 latent columns each: a decode batch has few rows.
  cudaError_t e = launch_head_gemm<128, 128, 2, 4>(qa_map, wuk_map, 0, 192, q_full,
                                                   static_cast<long long>(H) * 576, 576,
                                                   static_cast<const __nv_bfloat16*>(a.q) + 128,
                                                   static_cast<long long>(H) * 192, 192, T, H, a.status, stream);
  if (e != cudaSuccess) return e;

  // 2. Latent attention over the key partitions.
  const uint64_t cache_rows = static_cast<uint64_t>(a.num_pages) * a.page_size;
  CUtensorMap qr_map, kl_map, kr_map, kl1_map, kr1_map;
  if (!encode_2d(&qr_map, q_full, bf, 576, R, 1152, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode_2d(&kl_map, a.kv_cache, bf, 576, cache_rows, 1152, 64, DBN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&kr_map, a.kv_cache, bf, 576, cache_rows, 1152, 32, DBN, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode_2d(&kl1_map, a.kv_cache, bf, 576, cache_rows, 1152, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&kr1_map, a.kv_cache, bf, 576, cache_rows, 1152, 32, 1, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  DecodeParams p;
  p.q_full = q_full;
  p.iro = a.iro;
  p.cache_len = a.cache_len;
  p.page_table = a.page_table;
  p.indices = a.indices;
  p.topk = a.topk;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.indices_stride = a.indices_stride;
  p.num_pages = a.num_pages;
  p.page_size = a.page_size;
  p.max_pages = a.max_pages;
  p.B = a.B;
  p.H = H;
  p.R = static_cast<int>(R);
  p.parts = a.parts;
  p.part_keys = a.part_keys;
  p.m_tiles = static_cast<int>((static_cast<long long>(a.max_new) * H + 127) / 128);
  p.dense_tiles = (a.indices == nullptr && a.page_size % DBN == 0) ? 1 : 0;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  const long long total = static_cast<long long>(a.B) * a.parts * p.m_tiles;
  if (total > 0) {
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    const bool dense = p.dense_tiles != 0;
    const int clusters = dense ? decode_clusters<true>(dev) : decode_clusters<false>(dev);
    if (clusters <= 0) return cudaErrorInvalidConfiguration;
    const int grid = 2 * static_cast<int>(std::min<long long>(total, clusters));
    if (dense)
      e = launch_pdl(decode_attn_kernel<true>, dim3(grid), dim3(D_THREADS), D_SMEM_TOTAL, stream, qr_map, kl_map,
                     kr_map, kl1_map, kr1_map, p, static_cast<int>(total), static_cast<const uint8_t*>(a.kv_cache));
    else
      e = launch_pdl(decode_attn_kernel<false>, dim3(grid), dim3(D_THREADS), D_SMEM_TOTAL, stream, qr_map, kl_map,
                     kr_map, kl1_map, kr1_map, p, static_cast<int>(total), static_cast<const uint8_t*>(a.kv_cache));
    if (e != cudaSuccess) return e;
  }

  // 3. Merge the partitions (and the sink) into the bf16 latent result.
  const long long blocks = std::min<long long>((R + 3) / 4, 4ll * sm_count());
  if ((e = launch_pdl(decode_merge_kernel, dim3(static_cast<unsigned>(std::max(1ll, blocks))), dim3(256), 0, stream,
                      p, o_lat, a.lse, a.sink)) != cudaSuccess)
    return e;

  // 4. out = w_uv[h] o_lat.
  CUtensorMap ol_map, wuv_map;
  if (!encode_2d(&ol_map, o_lat, bf, static_cast<uint64_t>(H) * 512, T, static_cast<uint64_t>(H) * 1024, 64, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&wuv_map, a.w_uv, bf, 512, static_cast<uint64_t>(H) * 128, 1024, 64, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  return launch_head_gemm<128, 512, 4>(ol_map, wuv_map, 0, 512, static_cast<__nv_bfloat16*>(a.out),
                                       static_cast<long long>(H) * 128, 128, nullptr, 0, 0, T, H, a.status, stream);
}

}  // namespace mla
