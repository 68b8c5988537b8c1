// Chunk plan ("mla_prefill_plan" page): the context tokens of all sequences,
// cached first then new, laid end to end in batch order, are cut into chunks
// of S = buffer_token_size rows.  With P_b the exclusive prefix sum of the
// context lengths L_b and TOT their total, chunk c holds
//   buffer_row_offsets[c][b] = clamp(P_b - c*S, 0, S)        (b = 0..B)
//   cache_offsets[c][b]      = clamp(c*S - P_b, 0, L_b)      (b = 0..B-1)
//   buffer_lengths[c]        = c*S < TOT ? min(S, TOT - c*S) : -1
// so the whole plan is one prefix sum followed by independent writes.
//
// Small batches run in one CTA (warp-shuffle scan + a scan of warp totals);
// large batches run in two passes over tiles (described below).

#include "kernels.cuh"

namespace mla {

namespace {

constexpr int kThreads = 1024;
constexpr int kOneCtaMax = 4096;             // largest batch planned by a single CTA

__device__ __forceinline__ uint64_t clamp_u64(int64_t v, int64_t hi) {
  return static_cast<uint64_t>(v < 0 ? 0 : (v > hi ? hi : v));
}

// Context length of sequence b; flags malformed offsets.
__device__ __forceinline__ uint64_t ctx_len(const uint32_t* iro, const uint32_t* cache_len, int b,
                                            int& bad) {
  const uint32_t a = iro[b], e = iro[b + 1];
  if (e < a) {
    bad = 1;
    return cache_len[b];
  }
  return static_cast<uint64_t>(cache_len[b]) + (e - a);
}

// Inclusive block-wide scan of one value per thread (1024 threads).
__device__ __forceinline__ uint64_t block_scan(uint64_t v, uint64_t* warp_tot, uint64_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint64_t n = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint64_t w = warp_tot[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint64_t n = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += n;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const uint64_t before = warp ? warp_tot[warp - 1] : 0;
  total = warp_tot[31];
  __syncthreads();
  return v + before;
}

__device__ __forceinline__ void write_seq(uint32_t* bro, uint32_t* co, int B, int max_chunks,
                                          uint32_t S, int b, uint64_t excl, uint64_t L,
                                          bool skip_co_row0) {
  for (int c = 0; c < max_chunks; ++c) {
    const int64_t lo = static_cast<int64_t>(c) * S;
    bro[static_cast<size_t>(c) * (B + 1) + b] =
        static_cast<uint32_t>(clamp_u64(static_cast<int64_t>(excl) - lo, S));
    if (c > 0 || !skip_co_row0)
      co[static_cast<size_t>(c) * B + b] =
          static_cast<uint32_t>(clamp_u64(lo - static_cast<int64_t>(excl), static_cast<int64_t>(L)));
  }
}

__device__ __forceinline__ void write_tail(uint32_t* bro, int32_t* bl, int B, int max_chunks,
                                           uint32_t S, uint64_t tot, int bad, int32_t* status) {
  for (int c = threadIdx.x; c < max_chunks; c += blockDim.x) {
    const int64_t lo = static_cast<int64_t>(c) * S;
    const int64_t rest = static_cast<int64_t>(tot) - lo;
    bro[static_cast<size_t>(c) * (B + 1) + B] = static_cast<uint32_t>(clamp_u64(rest, S));
    bl[c] = rest > 0 ? static_cast<int32_t>(rest < S ? rest : S) : -1;
  }
  if (threadIdx.x == 0) {
    const uint64_t needed = (tot + S - 1) / S;
    if (bad || tot >= (1ull << 31))
      set_status(status, MLA_DEV_BAD_OFFSETS);
    else if (needed > static_cast<uint64_t>(max_chunks))
      set_status(status, MLA_DEV_TOO_MANY_CHUNKS);
  }
}

// One CTA walks the batch in tiles of 1024 sequences with a running carry.
__global__ void __launch_bounds__(kThreads) plan_one_cta(uint32_t* bro, uint32_t* co, int32_t* bl,
                                                         const uint32_t* iro,
                                                         const uint32_t* cache_len, int B,
                                                         int max_chunks, uint32_t S,
                                                         int32_t* status) {
  __shared__ uint64_t warp_tot[32];
  __shared__ int s_bad;
  pdl_enter();
  if (timed_out_before(status)) return;   // an earlier kernel timed out: no work
  if (threadIdx.x == 0) s_bad = (B >= 0 && iro[0] != 0) ? 1 : 0;
  __syncthreads();
  int bad = 0;
  uint64_t carry = 0;
  for (int base = 0; base < B; base += kThreads) {
    const int b = base + threadIdx.x;
    const uint64_t L = b < B ? ctx_len(iro, cache_len, b, bad) : 0;
    uint64_t tile_total;
    const uint64_t incl = block_scan(L, warp_tot, tile_total);
    if (b < B) write_seq(bro, co, B, max_chunks, S, b, carry + incl - L, L, false);
    carry += tile_total;
  }
  if (bad) atomicOr(&s_bad, 1);
  __syncthreads();
  write_tail(bro, bl, B, max_chunks, S, carry, s_bad, status);
}

// Large batches: two passes over tiles of 2048 sequences (256 threads, each
// lane of a warp owning 8 sequences strided by 32, so every load and store of
// a warp is one coalesced 128-byte access), with no CTA waiting for another:
//   pass A (plan_tile_totals)  each tile's total context length, stored in
//                              cache_offsets row 0, word 1 + t;
//   pass B (plan_tile_tables)  loads and scans its own sequences in registers
//                              (overlapping pass A: it is a programmatic
//                              dependent launch and waits for pass A only
//                              before it reads the totals), adds the totals of
//                              the tiles before it, and writes every table row
//                              chunk by chunk.
// Row 0 of cache_offsets is zero by definition, so it holds the scratch:
// word 0 counts finished pass-B tiles (zeroed by pass A), words 1..ntiles the
// tile totals (saturated to 32 bits).  No pass-B tile writes its row-0 entries
// there; the last pass-B tile to finish zeroes them, so row 0 ends all zero as
// the closed form says.  With TOT < 2^31 (anything larger is reported as bad
// offsets) every prefix fits in 32 bits, and so does the table arithmetic.
constexpr int kSThreads = 256;
constexpr int kSWarps = kSThreads / 32;
constexpr int kSPerLane = 8;
constexpr int kSTile = kSThreads * kSPerLane;   // 2048

__device__ __forceinline__ uint32_t sat32(uint64_t v) {
  return v > 0xFFFFFFFFull ? 0xFFFFFFFFu : static_cast<uint32_t>(v);
}

__device__ __forceinline__ uint64_t warp_sum64(uint64_t v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Block-wide sum of one 64-bit value per thread (every thread gets it).
__device__ __forceinline__ uint64_t block_sum64(uint64_t v, uint64_t* red) {
  v = warp_sum64(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  uint64_t s = 0;
#pragma unroll
  for (int w = 0; w < kSWarps; ++w) s += red[w];
  return s;
}

__global__ void __launch_bounds__(kSThreads) plan_tile_totals(uint32_t* co, const uint32_t* iro,
                                                              const uint32_t* cache_len, int B,
                                                              const int32_t* status) {
  __shared__ uint64_t red[kSWarps];
  // After the previous kernel of the stream, let pass B's CTAs start their
  // own loads while this pass runs.
  pdl_enter();
  if (timed_out_before(status)) return;   // pass B returns too
  const int t = blockIdx.x;
  const int base = t * kSTile;
  uint64_t v = 0;
#pragma unroll
  for (int k = 0; k < kSPerLane; ++k) {
    const int e = base + k * kSThreads + static_cast<int>(threadIdx.x);
    if (e < B) v += cache_len[e];
  }
  const uint64_t tot = block_sum64(v, red);
  if (threadIdx.x == 0) {
    // New tokens of the tile telescope to a difference of two offsets (a
    // decreasing pair is reported by pass B).
    const uint32_t a = iro[base], e = iro[min(base + kSTile, B)];
    co[1 + t] = sat32(tot + (e >= a ? e - a : 0u));
    if (t == 0) co[0] = 0u;
  }
}

__global__ void __launch_bounds__(kSThreads, 5) plan_tile_tables(uint32_t* bro, uint32_t* co, int32_t* bl,
                                                                 const uint32_t* iro,
                                                                 const uint32_t* cache_len, int B,
                                                                 int ntiles, int max_chunks, uint32_t S,
                                                                 int32_t* status) {
  __shared__ uint32_t warp_tot[kSWarps];
  __shared__ uint64_t red[kSWarps];
  __shared__ int s_last;
  // After a pipeline timeout recorded on this status word, neither pass does
  // any work (no pass writes that code, so both passes read the same value).
  if (timed_out_before(status)) return;
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = t * kSTile + warp * (32 * kSPerLane) + lane;   // this thread's first sequence
  const int nk = B > e0 ? min(kSPerLane, (B - e0 + 31) / 32) : 0;
  const uint32_t n_scratch = 1u + static_cast<uint32_t>(ntiles);

  // Context lengths and the warp-local exclusive scan of each 32-wide group.
  uint32_t L[kSPerLane], ex[kSPerLane];
  uint32_t run = 0;
  int bad = 0;
#pragma unroll
  for (int k = 0; k < kSPerLane; ++k) {
    const int e = e0 + k * 32;
    uint32_t l = 0;
    if (e < B) {
      const uint32_t a = iro[e], n = iro[e + 1];
      const uint64_t l64 = static_cast<uint64_t>(cache_len[e]) + (n >= a ? n - a : 0u);
      bad |= (n < a) | (l64 >= (1ull << 31));
      l = static_cast<uint32_t>(l64);
    }
    L[k] = l;
    uint32_t incl = l;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    ex[k] = run + incl - l;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) warp_tot[warp] = run;
  const int any_bad = __syncthreads_or(bad);

  // Pass A has completed (and its writes are visible) past this point.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  uint64_t pv = 0;
#pragma unroll 8
  for (int j = threadIdx.x; j < t; j += kSThreads) pv += __ldcg(co + 1 + j);
  const uint64_t prefix = block_sum64(pv, red);   // (its barrier also publishes warp_tot)

  if (t == ntiles - 1 && warp == 0) {
    // The last tile knows the total: the [c][B] column, buffer_lengths and
    // the status (2^31 tokens or more reads as bad offsets).
    const uint64_t tot = prefix + __ldcg(co + 1 + t);
    const bool bad_all = iro[0] != 0 || tot >= (1ull << 31);
    for (int c = lane; c < max_chunks; c += 32) {
      const int64_t lo = static_cast<int64_t>(c) * S;
      const int64_t rest = static_cast<int64_t>(tot) - lo;
      bro[static_cast<size_t>(c) * (B + 1) + B] = static_cast<uint32_t>(clamp_u64(rest, S));
      bl[c] = rest > 0 ? static_cast<int32_t>(rest < S ? rest : S) : -1;
    }
    if (lane == 0) {
      const uint64_t needed = (tot + S - 1) / S;
      if (bad_all)
        set_status(status, MLA_DEV_BAD_OFFSETS);
      else if (needed > static_cast<uint64_t>(max_chunks))
        set_status(status, MLA_DEV_TOO_MANY_CHUNKS);
    }
  }
  if (threadIdx.x == 0 && (any_bad || prefix >= (1ull << 31))) set_status(status, MLA_DEV_BAD_OFFSETS);

  // Every table row, chunk by chunk: with m = max(P_b, c*S),
  //   buffer_row_offsets = min(m - c*S, S),  cache_offsets = min(m - P_b, L_b).
  uint32_t off = static_cast<uint32_t>(prefix);
  for (int w = 0; w < warp; ++w) off += warp_tot[w];
#pragma unroll
  for (int k = 0; k < kSPerLane; ++k) ex[k] += off;
  uint32_t* br = bro + e0;
  uint32_t* cr = co + e0;
#pragma unroll
  for (int k = 0; k < kSPerLane; ++k) {
    if (k < nk) {
      br[32 * k] = min(ex[k], S);
      if (static_cast<uint32_t>(e0 + 32 * k) >= n_scratch) cr[32 * k] = 0u;
    }
  }
  uint64_t lo64 = S;
  for (int c = 1; c < max_chunks; ++c) {
    br += B + 1;
    cr += B;
    const uint32_t lo = sat32(lo64);
#pragma unroll
    for (int k = 0; k < kSPerLane; ++k) {
      if (k < nk) {
        const uint32_t m = max(ex[k], lo);
        br[32 * k] = min(m - lo, S);
        cr[32 * k] = min(m - ex[k], L[k]);
      }
    }
    lo64 += S;
  }

  // The last tile to finish zeroes the scratch (row 0 of cache_offsets).
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(co, 1u) == static_cast<uint32_t>(ntiles - 1);
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (uint32_t i = threadIdx.x; i < n_scratch; i += kSThreads) co[i] = 0u;
  }
}

}  // namespace

cudaError_t launch_plan(uint32_t* bro, uint32_t* co, int32_t* bl, const uint32_t* iro,
                        const uint32_t* cache_len, int B, int max_chunks, uint32_t S,
                        int32_t* status, cudaStream_t stream) {
  if (B <= kOneCtaMax) {
    return launch_pdl(plan_one_cta, dim3(1), dim3(kThreads), 0, stream, bro, co, bl, iro, cache_len, B, max_chunks,
                      S, status);
  }
  const int ntiles = (B + kSTile - 1) / kSTile;
  cudaError_t err = launch_pdl(plan_tile_totals, dim3(ntiles), dim3(kSThreads), 0, stream, co, iro, cache_len, B,
                               static_cast<const int32_t*>(status));
  if (err != cudaSuccess) return err;
  // Pass B as a programmatic dependent launch of pass A.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntiles);
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_tile_tables, bro, co, bl, iro, cache_len, B, ntiles, max_chunks, S,
                            status);
}

}  // namespace mla
