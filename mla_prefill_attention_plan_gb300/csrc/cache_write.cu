// Latent-cache write ("mla_prefill_decode_graph_bf16", Args freqs_cis,
// kv_norm_gamma, epsilon, kv_collection; Parameters kv_input_fn): the step in
// front of the prefill path.  New token i of sequence b (row
// input_row_offsets[b] + i of the latent rows and of q) sits at context
// position p = cache_lengths[b] + i.  Its 576 latent values are 512 c_kv
// values, normalised as x / sqrt(mean(x^2) + epsilon) * kv_norm_gamma, and 64
// k_rope values, rotated by freqs_cis[p] (32 complex numbers stored as
// interleaved (real, imaginary) pairs; the rotation is their complex product).
// The row, times the cache's inverse scale, is stored at page
// page_table[b][p / page_size], slot p % page_size, as bf16 or e4m3.  The rope
// part (last 64 values) of every head of q[row] is rotated in place by the same
// freqs_cis row.
//
// One CTA of 128 threads per token (grid-stride over tokens).  Thread j holds
// latent values 4j..4j+3 (one 8-byte load), so the sum of squares is a warp
// shuffle reduction plus four partials in shared memory; threads 0..15 rotate
// two k_rope pairs each; the q rope parts are 16-byte pieces of four pairs, 8
// per head, spread over the threads.  Every access of a warp is coalesced.
// HBM-bound: per token 1152 bytes of latent read, 576 * elt bytes of cache
// written, 256 bytes of frequencies read and 2 * H * 128 bytes of q read and
// written.
#include "kernels.cuh"

namespace mla {

namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// (re, im) * (c, s) as a complex product.
__device__ __forceinline__ float2 rotate(float re, float im, float c, float s) {
  return make_float2(fmaf(re, c, -im * s), fmaf(re, s, im * c));
}

template <int ELT>
__global__ void __launch_bounds__(kThreads)
    cache_write_kernel(uint8_t* __restrict__ kv_cache, uint16_t* __restrict__ q,
                       const uint16_t* __restrict__ kv_latent, const float* __restrict__ gamma,
                       const float* __restrict__ freqs, const uint32_t* __restrict__ iro,
                       const uint32_t* __restrict__ cache_len, const int32_t* __restrict__ page_table,
                       int num_pages, int page_size, int max_pages, int B, int H, int T,
                       int max_seq_len, float eps, float inv_scale, int32_t* status) {
  constexpr int kRowBytes = 576 * ELT;
  __shared__ float part[kThreads / 32];
  __shared__ int s_pos;
  __shared__ uint8_t* s_dst;
  if (timed_out_before(status)) return;   // an earlier kernel timed out: no work
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float4 g4 = reinterpret_cast<const float4*>(gamma)[tid];

  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (tid == 0) {
      // Largest b with iro[b] <= t; the token belongs to b when t < iro[b+1].
      int lo = 0, hi = B;   // search [lo, hi)
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (iro[mid] <= static_cast<uint32_t>(t)) lo = mid; else hi = mid;
      }
      int pos = -1;
      uint8_t* dst = nullptr;
      const uint32_t a = iro[lo], e = iro[lo + 1];
      if (a <= static_cast<uint32_t>(t) && static_cast<uint32_t>(t) < e) {
        const uint64_t p = static_cast<uint64_t>(cache_len[lo]) + (static_cast<uint32_t>(t) - a);
        if (p < static_cast<uint64_t>(max_seq_len)) {
          pos = static_cast<int>(p);
          const uint64_t pidx = p / static_cast<uint32_t>(page_size);
          const int page = pidx < static_cast<uint64_t>(max_pages)
                               ? page_table[static_cast<size_t>(lo) * max_pages + pidx] : -1;
          if (page >= 0 && page < num_pages)
            dst = kv_cache + (static_cast<size_t>(page) * page_size + p % page_size) * kRowBytes;
          else
            set_status(status, MLA_DEV_BAD_PAGE);
        } else {
          set_status(status, MLA_DEV_BAD_OFFSETS);
        }
      } else {
        set_status(status, MLA_DEV_BAD_OFFSETS);
      }
      s_pos = pos;
      s_dst = dst;
    }
    __syncthreads();
    const int pos = s_pos;
    uint8_t* const dst = s_dst;
    const float* fr = freqs + static_cast<size_t>(pos) * 64;

    // Latent: RMSNorm of the 512 c_kv values, then the 64 k_rope values.
    const uint16_t* row = kv_latent + static_cast<size_t>(t) * 576;
    const uint2 x = reinterpret_cast<const uint2*>(row)[tid];
    const float x0 = bf16_lo(x.x), x1 = bf16_hi(x.x), x2 = bf16_lo(x.y), x3 = bf16_hi(x.y);
    float ss = fmaf(x0, x0, fmaf(x1, x1, fmaf(x2, x2, x3 * x3)));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
    if (lane == 0) part[warp] = ss;
    __syncthreads();
    if (pos >= 0) {
      const float mean_sq = ((part[0] + part[1]) + (part[2] + part[3])) * (1.0f / 512.0f);
      const float r = 1.0f / sqrtf(mean_sq + eps) * inv_scale;
      const float y0 = x0 * r * g4.x, y1 = x1 * r * g4.y, y2 = x2 * r * g4.z, y3 = x3 * r * g4.w;
      if (dst != nullptr) {
        if (ELT == 2)
          reinterpret_cast<uint2*>(dst)[tid] = make_uint2(pack_bf16(y0, y1), pack_bf16(y2, y3));
        else
          reinterpret_cast<uint32_t*>(dst)[tid] =
              static_cast<uint32_t>(pack_e4m3(y0, y1)) | (static_cast<uint32_t>(pack_e4m3(y2, y3)) << 16);
      }
      if (tid < 16) {
        // k_rope values 4*tid .. 4*tid+3: pairs 2*tid and 2*tid+1.
        const uint2 k = reinterpret_cast<const uint2*>(row + 512)[tid];
        const float4 f = reinterpret_cast<const float4*>(fr)[tid];
        const float2 r0 = rotate(bf16_lo(k.x), bf16_hi(k.x), f.x, f.y);
        const float2 r1 = rotate(bf16_lo(k.y), bf16_hi(k.y), f.z, f.w);
        if (dst != nullptr) {
          if (ELT == 2)
            reinterpret_cast<uint2*>(dst + 1024)[tid] =
                make_uint2(pack_bf16(r0.x * inv_scale, r0.y * inv_scale), pack_bf16(r1.x * inv_scale, r1.y * inv_scale));
          else
            reinterpret_cast<uint32_t*>(dst + 512)[tid] =
                static_cast<uint32_t>(pack_e4m3(r0.x * inv_scale, r0.y * inv_scale)) |
                (static_cast<uint32_t>(pack_e4m3(r1.x * inv_scale, r1.y * inv_scale)) << 16);
        }
      }
      // q: piece m of head h holds rope values 8m .. 8m+7 (pairs 4m .. 4m+3).
      if (q != nullptr) {
        uint16_t* qt = q + static_cast<size_t>(t) * H * 192 + 128;
        for (int i = tid; i < 8 * H; i += kThreads) {
          const int h = i >> 3, m = i & 7;
          uint4* pq = reinterpret_cast<uint4*>(qt + static_cast<size_t>(h) * 192) + m;
          const uint4 v = *pq;
          const float4 fa = reinterpret_cast<const float4*>(fr)[2 * m];
          const float4 fb = reinterpret_cast<const float4*>(fr)[2 * m + 1];
          const float2 a0 = rotate(bf16_lo(v.x), bf16_hi(v.x), fa.x, fa.y);
          const float2 a1 = rotate(bf16_lo(v.y), bf16_hi(v.y), fa.z, fa.w);
          const float2 a2 = rotate(bf16_lo(v.z), bf16_hi(v.z), fb.x, fb.y);
          const float2 a3 = rotate(bf16_lo(v.w), bf16_hi(v.w), fb.z, fb.w);
          *pq = make_uint4(pack_bf16(a0.x, a0.y), pack_bf16(a1.x, a1.y), pack_bf16(a2.x, a2.y),
                           pack_bf16(a3.x, a3.y));
        }
      }
    }
    __syncthreads();   // s_pos, s_dst and part are rewritten for the next token
  }
}

}  // namespace

cudaError_t launch_cache_write(const CacheWriteArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  const int grid = a.T < 16 * sm_count() ? a.T : 16 * sm_count();
  if (a.elt_bytes == 2)
    cache_write_kernel<2><<<grid, kThreads, 0, stream>>>(
        static_cast<uint8_t*>(a.kv_cache), static_cast<uint16_t*>(a.q), static_cast<const uint16_t*>(a.kv_latent),
        a.gamma, a.freqs, a.iro, a.cache_len, a.page_table, a.num_pages, a.page_size, a.max_pages, a.B, a.H, a.T,
        a.max_seq_len, a.eps, a.inv_scale, a.status);
  else
    cache_write_kernel<1><<<grid, kThreads, 0, stream>>>(
        static_cast<uint8_t*>(a.kv_cache), static_cast<uint16_t*>(a.q), static_cast<const uint16_t*>(a.kv_latent),
        a.gamma, a.freqs, a.iro, a.cache_len, a.page_table, a.num_pages, a.page_size, a.max_pages, a.B, a.H, a.T,
        a.max_seq_len, a.eps, a.inv_scale, a.status);
  return cudaGetLastError();
}

}  // namespace mla
