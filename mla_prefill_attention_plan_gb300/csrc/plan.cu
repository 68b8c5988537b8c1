// Chunk plan ("mla_prefill_plan" page): the context tokens of all sequences,
// cached first then new, laid end to end in batch order, are cut into chunks
// of S = buffer_token_size rows.  With P_b the exclusive prefix sum of the
// context lengths L_b and TOT their total, chunk c holds
//   buffer_row_offsets[c][b] = clamp(P_b - c*S, 0, S)        (b = 0..B)
//   cache_offsets[c][b]      = clamp(c*S - P_b, 0, L_b)      (b = 0..B-1)
//   buffer_lengths[c]        = c*S < TOT ? min(S, TOT - c*S) : -1
// so the whole plan is one prefix sum followed by independent writes.
//
// Small batches run in one CTA (warp-shuffle scan + a scan of warp totals).
// Large batches run in two passes over many CTAs; the per-CTA totals of the
// first pass are parked in row 0 of cache_offsets (which the plan defines to
// be all zeros) and that row is cleared at the end.
#include "kernels.cuh"

namespace mla {

namespace {

constexpr int kThreads = 1024;
constexpr int kItems = 4;                    // sequences per thread in the multi-CTA pass
constexpr int kTile = kThreads * kItems;     // sequences per CTA in the multi-CTA pass

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

// Pass 1 of the multi-CTA plan: per-CTA totals into cache_offsets row 0.
__global__ void __launch_bounds__(kThreads) plan_tile_sums(uint32_t* co_row0, const uint32_t* iro,
                                                           const uint32_t* cache_len, int B) {
  __shared__ uint64_t warp_tot[32];
  int bad = 0;
  uint64_t v = 0;
  const int base = blockIdx.x * kTile;
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int b = base + k * kThreads + threadIdx.x;
    if (b < B) v += ctx_len(iro, cache_len, b, bad);
  }
  uint64_t total;
  block_scan(v, warp_tot, total);
  // Totals fit in 32 bits whenever the whole batch is below 2^31 tokens (larger
  // batches are rejected by pass 2); saturate so an oversize tile still shows.
  if (threadIdx.x == 0) co_row0[blockIdx.x] = total > 0xFFFFFFFFull ? 0xFFFFFFFFu : uint32_t(total);
}

// Pass 2: every CTA adds up the totals of the CTAs before it, scans its own
// tile and writes every table entry except cache_offsets row 0.
__global__ void __launch_bounds__(kThreads) plan_tile_write(uint32_t* bro, uint32_t* co, int32_t* bl,
                                                            const uint32_t* iro,
                                                            const uint32_t* cache_len, int B,
                                                            int max_chunks, uint32_t S,
                                                            int32_t* status) {
  __shared__ uint64_t warp_tot[32];
  __shared__ int s_bad;
  const int ntiles = gridDim.x;
  // Sum of the tile totals before this CTA, and of all of them.
  uint64_t before = 0, all = 0;
  for (int t = threadIdx.x; t < ntiles; t += kThreads) {
    const uint64_t s = co[t];
    all += s;
    if (t < static_cast<int>(blockIdx.x)) before += s;
  }
  uint64_t before_sum, all_sum;
  block_scan(before, warp_tot, before_sum);
  block_scan(all, warp_tot, all_sum);
  if (threadIdx.x == 0) s_bad = iro[0] != 0 ? 1 : 0;
  __syncthreads();
  int bad = 0;
  uint64_t carry = before_sum;
  const int base = blockIdx.x * kTile;
  for (int k = 0; k < kItems; ++k) {
    const int b = base + k * kThreads + threadIdx.x;
    const uint64_t L = b < B ? ctx_len(iro, cache_len, b, bad) : 0;
    uint64_t tile_total;
    const uint64_t incl = block_scan(L, warp_tot, tile_total);
    if (b < B) write_seq(bro, co, B, max_chunks, S, b, carry + incl - L, L, true);
    carry += tile_total;
  }
  if (bad) atomicOr(&s_bad, 1);
  __syncthreads();
  if (blockIdx.x == 0) write_tail(bro, bl, B, max_chunks, S, all_sum, s_bad, status);
  else if (s_bad && threadIdx.x == 0) set_status(status, MLA_DEV_BAD_OFFSETS);
}

}  // namespace

cudaError_t launch_plan(uint32_t* bro, uint32_t* co, int32_t* bl, const uint32_t* iro,
                        const uint32_t* cache_len, int B, int max_chunks, uint32_t S,
                        int32_t* status, cudaStream_t stream) {
  if (B <= kTile) {
    plan_one_cta<<<1, kThreads, 0, stream>>>(bro, co, bl, iro, cache_len, B, max_chunks, S, status);
    return cudaGetLastError();
  }
  const int ntiles = (B + kTile - 1) / kTile;
  plan_tile_sums<<<ntiles, kThreads, 0, stream>>>(co, iro, cache_len, B);
  plan_tile_write<<<ntiles, kThreads, 0, stream>>>(bro, co, bl, iro, cache_len, B, max_chunks, S,
                                                   status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // Row 0 of cache_offsets is all zeros by definition (chunk 0 starts every
  // sequence at position 0); it held the tile totals until now.
  return cudaMemsetAsync(co, 0, sizeof(uint32_t) * static_cast<size_t>(B), stream);
}

}  // namespace mla
