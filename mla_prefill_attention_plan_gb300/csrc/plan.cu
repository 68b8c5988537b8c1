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
// large batches run in three passes over tiles (described below).
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

// Large batches: three passes over tiles of 4096 sequences (256 threads, each
// lane of a warp owning 16 sequences strided by 32, so every load and store of
// a warp is one coalesced 128-byte access).
//   pass 1  per-tile total of the context lengths, parked in the tile's own
//           first entry of cache_offsets row 0 (that row is zero by definition
//           and is rewritten by pass 3);
//   pass 2  one CTA turns the parked totals into exclusive tile prefixes in
//           place and writes buffer_lengths, the [c][B] column and the status;
//   pass 3  every tile reads its own prefix, scans its sequences with warp
//           shuffles and writes its part of every table row (row 0 of
//           cache_offsets comes out zero, overwriting the parked value).
constexpr int kWThreads = 256;
constexpr int kWPerLane = 16;
constexpr int kWTile = kWThreads * kWPerLane;   // 4096

__device__ __forceinline__ int tile_elem(int base, int warp, int lane, int k) {
  return base + warp * (32 * kWPerLane) + k * 32 + lane;
}

__global__ void __launch_bounds__(kWThreads) plan_tile_sums(uint32_t* co_row0, const uint32_t* iro,
                                                            const uint32_t* cache_len, int B) {
  __shared__ uint64_t warp_sum[kWThreads / 32];
  const int base = blockIdx.x * kWTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t v = 0;
#pragma unroll
  for (int k = 0; k < kWPerLane; ++k) {
    const int e = tile_elem(base, warp, lane, k);
    if (e < B) v += cache_len[e];
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_down_sync(0xffffffffu, v, d);
  if (lane == 0) warp_sum[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t t = 0;
    for (int w = 0; w < kWThreads / 32; ++w) t += warp_sum[w];
    // New tokens of the tile telescope to a difference of two offsets (a
    // decreasing pair is reported by pass 3; clamp so the sum stays sane).
    const int end = min(base + kWTile, B);
    const uint32_t a = iro[base], e = iro[end];
    t += e >= a ? (e - a) : 0;
    co_row0[base] = t > 0xFFFFFFFFull ? 0xFFFFFFFFu : static_cast<uint32_t>(t);
  }
}

__global__ void __launch_bounds__(kThreads) plan_tile_scan(uint32_t* bro, uint32_t* co_row0,
                                                           int32_t* bl, const uint32_t* iro, int B,
                                                           int max_chunks, uint32_t S,
                                                           int32_t* status) {
  __shared__ uint64_t warp_tot[32];
  const int ntiles = (B + kWTile - 1) / kWTile;
  uint64_t carry = 0;
  for (int t0 = 0; t0 < ntiles; t0 += kThreads) {
    const int t = t0 + threadIdx.x;
    const uint64_t v = t < ntiles ? co_row0[static_cast<size_t>(t) * kWTile] : 0;
    uint64_t round_total;
    const uint64_t incl = block_scan(v, warp_tot, round_total);
    if (t < ntiles) {
      const uint64_t excl = carry + incl - v;
      co_row0[static_cast<size_t>(t) * kWTile] = excl > 0xFFFFFFFFull ? 0xFFFFFFFFu : uint32_t(excl);
    }
    carry += round_total;
  }
  write_tail(bro, bl, B, max_chunks, S, carry, iro[0] != 0, status);
}

__global__ void __launch_bounds__(kWThreads) plan_tile_write(uint32_t* bro, uint32_t* co, const uint32_t* iro,
                                                             const uint32_t* cache_len, int B,
                                                             int max_chunks, uint32_t S,
                                                             int32_t* status) {
  __shared__ uint64_t warp_sum[kWThreads / 32];
  __shared__ uint64_t tile_prefix;
  const int base = blockIdx.x * kWTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) tile_prefix = co[base];   // parked by pass 2
  uint32_t L[kWPerLane];
  int bad = 0;
  uint64_t mine = 0;
#pragma unroll
  for (int k = 0; k < kWPerLane; ++k) {
    const int e = tile_elem(base, warp, lane, k);
    uint32_t l = 0;
    if (e < B) {
      const uint32_t a = iro[e], n = iro[e + 1];
      if (n < a) bad = 1;
      l = cache_len[e] + (n >= a ? n - a : 0u);
    }
    L[k] = l;
    mine += l;
  }
  uint64_t wsum = mine;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, d);
  if (lane == 0) warp_sum[warp] = wsum;
  __syncthreads();   // also orders every read of the parked prefix before row 0 is rewritten
  uint64_t carry = tile_prefix;
  for (int w = 0; w < warp; ++w) carry += warp_sum[w];
#pragma unroll
  for (int k = 0; k < kWPerLane; ++k) {
    const int e = tile_elem(base, warp, lane, k);
    uint64_t incl = L[k];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint64_t n = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += n;
    }
    const uint64_t excl = carry + incl - L[k];
    carry += __shfl_sync(0xffffffffu, incl, 31);
    if (e < B) {
      for (int c = 0; c < max_chunks; ++c) {
        const int64_t lo = static_cast<int64_t>(c) * S;
        bro[static_cast<size_t>(c) * (B + 1) + e] =
            static_cast<uint32_t>(clamp_u64(static_cast<int64_t>(excl) - lo, S));
        co[static_cast<size_t>(c) * B + e] =
            static_cast<uint32_t>(clamp_u64(lo - static_cast<int64_t>(excl), static_cast<int64_t>(L[k])));
      }
    }
  }
  if (bad) set_status(status, MLA_DEV_BAD_OFFSETS);
}

}  // namespace

cudaError_t launch_plan(uint32_t* bro, uint32_t* co, int32_t* bl, const uint32_t* iro,
                        const uint32_t* cache_len, int B, int max_chunks, uint32_t S,
                        int32_t* status, cudaStream_t stream) {
  if (B <= kOneCtaMax) {
    plan_one_cta<<<1, kThreads, 0, stream>>>(bro, co, bl, iro, cache_len, B, max_chunks, S, status);
    return cudaGetLastError();
  }
  const int ntiles = (B + kWTile - 1) / kWTile;
  plan_tile_sums<<<ntiles, kWThreads, 0, stream>>>(co, iro, cache_len, B);
  plan_tile_scan<<<1, kThreads, 0, stream>>>(bro, co, bl, iro, B, max_chunks, S, status);
  plan_tile_write<<<ntiles, kWThreads, 0, stream>>>(bro, co, iro, cache_len, B, max_chunks, S, status);
  return cudaGetLastError();
}

}  // namespace mla
