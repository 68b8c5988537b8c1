// Latent gather ("mla_prefill_decode_graph_bf16", Parameters: kv_input_fn;
// "flare_mla_prefill_dispatch", Parameters: k_rope_t): copy one plan chunk's
// context tokens out of the paged cache into contiguous buffers.
//
// Buffer row r of chunk c belongs to the sequence b with
// buffer_row_offsets[c][b] <= r < buffer_row_offsets[c][b+1]; it is the cache
// token at context position p = cache_offsets[c][b] + (r - buffer_row_offsets
// [c][b]), stored in page page_table[b][p / page_size], slot p % page_size.
// The 576-element cache row splits into 512 latent values (c_kv_buf) and 64
// rope values (k_rope_buf).
//
// Each CTA owns 32 consecutive buffer rows: 32 threads first resolve the rows'
// source addresses (binary search over the chunk's row offsets, page-table
// lookup), then all 256 threads move the rows as 16-byte vectors with every
// thread keeping several loads in flight.  Consecutive threads touch
// consecutive 16-byte pieces of a row, and the rows of one page are adjacent
// in the cache, so reads and writes are coalesced.
#include "kernels.cuh"

namespace mla {

namespace {

constexpr int kRows = 32;
constexpr int kThreads = 256;

template <int ELT>
__global__ void __launch_bounds__(kThreads)
    gather_kernel(uint8_t* __restrict__ ckv_buf, uint8_t* __restrict__ krope_buf,
                  const uint8_t* __restrict__ cache, const int32_t* __restrict__ page_table,
                  int num_pages, int page_size, int max_pages, const uint32_t* __restrict__ bro,
                  const uint32_t* __restrict__ co, const int32_t* __restrict__ bl, int chunk, int B,
                  int S, int32_t* status) {
  constexpr int kRowBytes = 576 * ELT;
  constexpr int kVecPerRow = kRowBytes / 16;        // 72 (bf16) or 36 (e4m3)
  constexpr int kCkvVec = 512 * ELT / 16;           // 64 or 32
  constexpr int kRopeBytes = 64 * ELT;              // 128 or 64
  constexpr int kVecs = kRows * kVecPerRow;
  constexpr int kPerThread = (kVecs + kThreads - 1) / kThreads;

  __shared__ const uint8_t* src_row[kRows];
  pdl_enter();
  if (timed_out_before(status)) return;   // an earlier kernel timed out: no work
  const int n = min(bl[chunk], S);        // never past the buffers, whatever the table says
  const int r0 = blockIdx.x * kRows;
  if (r0 >= n) return;
  const uint32_t* bro_c = bro + static_cast<size_t>(chunk) * (B + 1);
  const uint32_t* co_c = co + static_cast<size_t>(chunk) * B;

  if (threadIdx.x < kRows) {
    const int r = r0 + threadIdx.x;
    const uint8_t* src = nullptr;
    if (r < n) {
      // Largest b with bro_c[b] <= r (rows of b then end after r).
      int lo = 0, hi = B;  // invariant: bro_c[lo] <= r < bro_c[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (bro_c[mid] <= static_cast<uint32_t>(r)) lo = mid; else hi = mid;
      }
      const uint32_t pos = co_c[lo] + (static_cast<uint32_t>(r) - bro_c[lo]);
      const uint32_t pidx = pos / static_cast<uint32_t>(page_size);
      const int page = pidx < static_cast<uint32_t>(max_pages)
                           ? page_table[static_cast<size_t>(lo) * max_pages + pidx] : -1;
      if (page >= 0 && page < num_pages)
        src = cache + (static_cast<size_t>(page) * page_size + pos % page_size) * kRowBytes;
      else
        set_status(status, MLA_DEV_BAD_PAGE);
    }
    src_row[threadIdx.x] = src;
  }
  __syncthreads();

  int4 v[kPerThread];
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int idx = threadIdx.x + k * kThreads;
    const int row = idx / kVecPerRow, col = idx - row * kVecPerRow;
    const uint8_t* src = idx < kVecs ? src_row[row] : nullptr;
    if (src != nullptr) v[k] = __ldg(reinterpret_cast<const int4*>(src) + col);
  }
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int idx = threadIdx.x + k * kThreads;
    const int row = idx / kVecPerRow, col = idx - row * kVecPerRow;
    const uint8_t* src = idx < kVecs ? src_row[row] : nullptr;
    if (src == nullptr) continue;
    const size_t r = static_cast<size_t>(r0 + row);
    if (col < kCkvVec)
      reinterpret_cast<int4*>(ckv_buf + r * (512 * ELT))[col] = v[k];
    else
      reinterpret_cast<int4*>(krope_buf + r * kRopeBytes)[col - kCkvVec] = v[k];
  }
}

// Cache-row table of the plan's chunks: cache_rows[c][r] = the cache row
// holding buffer row r of chunk c (the same lookup as above, 4 bytes per row
// instead of the row itself), 0 for r >= buffer_lengths[c] and for a row
// whose page is out of range (reported).  One thread per (chunk, row).
__global__ void __launch_bounds__(256)
    cache_rows_kernel(int32_t* __restrict__ cache_rows, const int32_t* __restrict__ page_table,
                      int num_pages, int page_size, int max_pages, const uint32_t* __restrict__ bro,
                      const uint32_t* __restrict__ co, const int32_t* __restrict__ bl, int B, int S,
                      int32_t* status) {
  if (timed_out_before(status)) return;
  const int chunk = blockIdx.y;
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= S) return;
  const int n = min(__ldg(bl + chunk), S);
  int row = 0;
  if (r < n) {
    const uint32_t* bro_c = bro + static_cast<size_t>(chunk) * (B + 1);
    const uint32_t* co_c = co + static_cast<size_t>(chunk) * B;
    int lo = 0, hi = B;  // invariant: bro_c[lo] <= r < bro_c[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(bro_c + mid) <= static_cast<uint32_t>(r)) lo = mid; else hi = mid;
    }
    const uint32_t pos = __ldg(co_c + lo) + (static_cast<uint32_t>(r) - __ldg(bro_c + lo));
    const uint32_t pidx = pos / static_cast<uint32_t>(page_size);
    const int page = pidx < static_cast<uint32_t>(max_pages)
                         ? __ldg(page_table + static_cast<size_t>(lo) * max_pages + pidx) : -1;
    if (page >= 0 && page < num_pages)
      row = static_cast<int>(static_cast<long long>(page) * page_size + pos % page_size);
    else
      set_status(status, MLA_DEV_BAD_PAGE);
  }
  cache_rows[static_cast<size_t>(chunk) * S + r] = row;
}

}  // namespace

cudaError_t launch_cache_rows(int32_t* cache_rows, const int32_t* page_table, int num_pages,
                              int page_size, int max_pages, const uint32_t* bro, const uint32_t* co,
                              const int32_t* bl, int max_chunks, int B, uint32_t S, int32_t* status,
                              cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((static_cast<uint64_t>(S) + 255) / 256), static_cast<unsigned>(max_chunks));
  cache_rows_kernel<<<grid, 256, 0, stream>>>(cache_rows, page_table, num_pages, page_size, max_pages, bro, co,
                                               bl, B, static_cast<int>(S), status);
  return cudaGetLastError();
}

cudaError_t launch_gather(void* c_kv_buf, void* k_rope_buf, const void* kv_cache,
                          const int32_t* page_table, int num_pages, int page_size, int max_pages,
                          const uint32_t* bro, const uint32_t* co, const int32_t* bl, int chunk,
                          int B, uint32_t S, int elt_bytes, int32_t* status, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((static_cast<uint64_t>(S) + kRows - 1) / kRows);
  if (elt_bytes == 2)
    return launch_pdl(gather_kernel<2>, dim3(grid), dim3(kThreads), 0, stream, static_cast<uint8_t*>(c_kv_buf),
                      static_cast<uint8_t*>(k_rope_buf), static_cast<const uint8_t*>(kv_cache), page_table,
                      num_pages, page_size, max_pages, bro, co, bl, chunk, B, static_cast<int>(S), status);
  return launch_pdl(gather_kernel<1>, dim3(grid), dim3(kThreads), 0, stream, static_cast<uint8_t*>(c_kv_buf),
                    static_cast<uint8_t*>(k_rope_buf), static_cast<const uint8_t*>(kv_cache), page_table,
                    num_pages, page_size, max_pages, bro, co, bl, chunk, B, static_cast<int>(S), status);
}

}  // namespace mla
