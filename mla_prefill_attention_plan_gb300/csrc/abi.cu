// C ABI of the library (declared in include/mla_prefill.h): argument checks,
// tensor-map encoding, workspace layout and the fused chunk loop.  No entry
// point allocates memory or synchronises the stream.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "kernels.cuh"

namespace mla {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int elt_bytes(int32_t dtype) { return dtype == MLA_BF16 ? 2 : 1; }

bool dtype_ok(int32_t dtype) { return dtype == MLA_BF16 || dtype == MLA_E4M3; }

mla_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_LAUNCH; }

// Workspace layout of the fused entry point.
struct Layout {
  size_t bro, co, bl, ckv, krope, knope, v, oacc, lseacc, total;
};

Layout layout(int B, int H, int T_q, int max_chunks, uint32_t S, int dtype) {
  const size_t e = elt_bytes(dtype);
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  L.bro = take(sizeof(uint32_t) * size_t(max_chunks) * (B + 1));
  L.co = take(sizeof(uint32_t) * size_t(max_chunks) * (B > 0 ? B : 1));
  L.bl = take(sizeof(int32_t) * size_t(max_chunks));
  L.ckv = take(size_t(S) * 512 * e);
  L.krope = take(size_t(S) * 64 * e);
  L.knope = take(size_t(S) * H * 128 * e);
  L.v = take(size_t(S) * H * 128 * 2);   // bf16, or f16 holding e4m3-rounded values
  const bool merge = max_chunks > 1;
  L.oacc = take(merge ? size_t(T_q) * H * 128 * sizeof(float) : 0);
  L.lseacc = take(merge ? size_t(T_q) * H * sizeof(float) : 0);
  L.total = off;
  return L;
}

}  // namespace

bool encode_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, uint64_t inner,
               uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || inner == 0 || outer == 0) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estride[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_string(int32_t code) {
  switch (code) {
    case MLA_OK: return "ok";
    case MLA_ERR_ARG: return "bad argument (null or misaligned pointer, or bad size)";
    case MLA_ERR_GEOMETRY: return "unsupported geometry";
    case MLA_ERR_DTYPE: return "unsupported dtype (bf16 or e4m3 only)";
    case MLA_ERR_LAUNCH: return "CUDA launch or tensor-map error";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_DEV_TOO_MANY_CHUNKS: return "device: plan needs more than max_chunks chunks";
    case MLA_DEV_BAD_OFFSETS: return "device: malformed input_row_offsets or lengths";
    case MLA_DEV_BAD_PAGE: return "device: page id out of range";
    case MLA_DEV_TIMEOUT: return "device: pipeline wait timed out";
    default: return "unknown status";
  }
}

int32_t mla_abi_version(void) { return MLA_ABI_VERSION; }

const char* mla_attention_kernel(int32_t dtype) {
  if (dtype == MLA_E4M3) return "e4m3";
  if (dtype != MLA_BF16) return nullptr;
  return "pair";
}

mla_status_t mla_selftest_bounded_wait(int32_t* d_status, int64_t* d_elapsed_ns, int64_t limit_ns,
                                       int32_t cluster_size, mla_stream_t stream) {
  if (!d_status || !d_elapsed_ns || (reinterpret_cast<uintptr_t>(d_elapsed_ns) & 7u) ||
      (cluster_size != 1 && cluster_size != 2) || limit_ns < 1000 ||
      limit_ns > static_cast<int64_t>(mla::kWaitLimitNs))
    return MLA_ERR_ARG;
  return from_cuda(mla::launch_bounded_wait_selftest(d_status, reinterpret_cast<long long*>(d_elapsed_ns),
                                                     static_cast<uint64_t>(limit_ns), cluster_size,
                                                     static_cast<cudaStream_t>(stream)));
}

mla_status_t mla_latent_cache_write(void* kv_cache, void* q, const void* kv_latent,
                                    const float* kv_norm_gamma, const float* freqs_cis,
                                    const uint32_t* input_row_offsets,
                                    const uint32_t* cache_lengths, const int32_t* page_table,
                                    int32_t num_pages, int32_t page_size,
                                    int32_t max_pages_per_seq, int32_t batch_size,
                                    int32_t num_heads, int32_t total_q_tokens,
                                    int32_t max_seq_len, float epsilon, float kv_inv_scale,
                                    int32_t dtype, int32_t* d_status, mla_stream_t stream) {
  if (!dtype_ok(dtype)) return MLA_ERR_DTYPE;
  if (!kv_cache || !kv_latent || !kv_norm_gamma || !freqs_cis || !input_row_offsets ||
      !cache_lengths || !page_table || !aligned16(kv_cache) || !aligned16(kv_latent) ||
      !aligned16(kv_norm_gamma) || !aligned16(freqs_cis) || (q && !aligned16(q)) ||
      batch_size < 1 || total_q_tokens < 0 || (q && num_heads < 1) || num_pages < 1 ||
      page_size < 1 || max_pages_per_seq < 1 || max_seq_len < 1 || !(epsilon >= 0.0f) ||
      !(kv_inv_scale > 0.0f))
    return MLA_ERR_ARG;
  mla::CacheWriteArgs a;
  a.kv_cache = kv_cache;
  a.q = q;
  a.kv_latent = kv_latent;
  a.gamma = kv_norm_gamma;
  a.freqs = freqs_cis;
  a.iro = input_row_offsets;
  a.cache_len = cache_lengths;
  a.page_table = page_table;
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.max_pages = max_pages_per_seq;
  a.B = batch_size;
  a.H = q ? num_heads : 0;
  a.T = total_q_tokens;
  a.max_seq_len = max_seq_len;
  a.eps = epsilon;
  a.inv_scale = kv_inv_scale;
  a.elt_bytes = elt_bytes(dtype);
  a.status = d_status;
  return from_cuda(mla::launch_cache_write(a, static_cast<cudaStream_t>(stream)));
}

mla_status_t mla_prefill_plan(uint32_t* buffer_row_offsets, uint32_t* cache_offsets,
                              int32_t* buffer_lengths, const uint32_t* input_row_offsets,
                              const uint32_t* cache_lengths, int32_t batch_size,
                              int32_t max_chunks, uint32_t buffer_token_size, int32_t* d_status,
                              mla_stream_t stream) {
  if (!buffer_row_offsets || !buffer_lengths || !input_row_offsets || batch_size < 0 ||
      max_chunks < 1 || buffer_token_size == 0)
    return MLA_ERR_ARG;
  if (batch_size > 0 && (!cache_offsets || !cache_lengths)) return MLA_ERR_ARG;
  return from_cuda(launch_plan(buffer_row_offsets, cache_offsets, buffer_lengths, input_row_offsets,
                               cache_lengths, batch_size, max_chunks, buffer_token_size, d_status,
                               static_cast<cudaStream_t>(stream)));
}

mla_status_t mla_gather_latent(void* c_kv_buf, void* k_rope_buf, const void* kv_cache,
                               const int32_t* page_table, int32_t num_pages, int32_t page_size,
                               int32_t max_pages_per_seq, const uint32_t* buffer_row_offsets,
                               const uint32_t* cache_offsets, const int32_t* buffer_lengths,
                               int32_t chunk, int32_t batch_size, uint32_t buffer_token_size,
                               int32_t dtype, int32_t* d_status, mla_stream_t stream) {
  if (!dtype_ok(dtype)) return MLA_ERR_DTYPE;
  if (!c_kv_buf || !k_rope_buf || !kv_cache || !page_table || !buffer_row_offsets ||
      !cache_offsets || !buffer_lengths || !aligned16(c_kv_buf) || !aligned16(k_rope_buf) ||
      !aligned16(kv_cache) || num_pages < 1 || page_size < 1 || max_pages_per_seq < 1 ||
      chunk < 0 || batch_size < 1 || buffer_token_size == 0)
    return MLA_ERR_ARG;
  return from_cuda(launch_gather(c_kv_buf, k_rope_buf, kv_cache, page_table, num_pages, page_size,
                                 max_pages_per_seq, buffer_row_offsets, cache_offsets,
                                 buffer_lengths, chunk, batch_size, buffer_token_size,
                                 elt_bytes(dtype), d_status, static_cast<cudaStream_t>(stream)));
}

mla_status_t mla_chunk_cache_rows(int32_t* cache_rows, const int32_t* page_table,
                                  int32_t num_pages, int32_t page_size, int32_t max_pages_per_seq,
                                  const uint32_t* buffer_row_offsets, const uint32_t* cache_offsets,
                                  const int32_t* buffer_lengths, int32_t max_chunks,
                                  int32_t batch_size, uint32_t buffer_token_size, int32_t* d_status,
                                  mla_stream_t stream) {
  if (!cache_rows || !page_table || !buffer_row_offsets || !cache_offsets || !buffer_lengths ||
      num_pages < 1 || page_size < 1 || max_pages_per_seq < 1 || max_chunks < 1 ||
      max_chunks > 65535 || batch_size < 1 || buffer_token_size == 0 ||
      buffer_token_size > 0x7FFFFFFFu || static_cast<int64_t>(num_pages) * page_size > 0x7FFFFFFFll)
    return MLA_ERR_ARG;
  return from_cuda(launch_cache_rows(cache_rows, page_table, num_pages, page_size, max_pages_per_seq,
                                     buffer_row_offsets, cache_offsets, buffer_lengths, max_chunks,
                                     batch_size, buffer_token_size, d_status,
                                     static_cast<cudaStream_t>(stream)));
}

// A rows from the c_kv buffer, or (kv_cache given) from the cache rows the
// chunk's table names.
static mla_status_t upproject_impl(void* k_nope, void* v, const void* c_kv_buf,
                                   const void* kv_cache, const int32_t* cache_rows,
                                   int32_t num_cache_rows, const void* w_k, const void* w_uv,
                                   const int32_t* buffer_lengths, int32_t chunk,
                                   uint32_t buffer_token_size, int32_t num_heads, int32_t dtype,
                                   float ckv_scale, float w_scale, float kv_out_inv_scale,
                                   int32_t* d_status, mla_stream_t stream) {
  if (!dtype_ok(dtype)) return MLA_ERR_DTYPE;
  if (num_heads < 1) return MLA_ERR_GEOMETRY;
  if (!k_nope || !v || !w_k || !w_uv || !aligned16(k_nope) || !aligned16(v) || !aligned16(w_k) ||
      !aligned16(w_uv) || chunk < 0 || buffer_token_size == 0 || buffer_token_size > 0x7FFFFFFFu)
    return MLA_ERR_ARG;
  if (kv_cache) {
    if (!aligned16(kv_cache) || !cache_rows || !buffer_lengths || num_cache_rows < 1) return MLA_ERR_ARG;
  } else if (!c_kv_buf || !aligned16(c_kv_buf)) {
    return MLA_ERR_ARG;
  }
  UpprojArgs a;
  a.kv_cache = kv_cache;
  a.cache_rows = cache_rows;
  a.num_cache_rows = num_cache_rows;
  a.k_nope = k_nope;
  a.v = v;
  a.c_kv = c_kv_buf;
  a.w_k = w_k;
  a.w_uv = w_uv;
  a.buffer_lengths = buffer_lengths;
  a.chunk = chunk;
  a.S = buffer_token_size;
  a.H = num_heads;
  a.dtype = dtype;
  a.out_scale = ckv_scale * w_scale * kv_out_inv_scale;
  a.status = d_status;
  return from_cuda(launch_upproject(a, static_cast<cudaStream_t>(stream)));
}

mla_status_t mla_upproject(void* k_nope, void* v, const void* c_kv_buf, const void* w_k,
                           const void* w_uv, const int32_t* buffer_lengths, int32_t chunk,
                           uint32_t buffer_token_size, int32_t num_heads, int32_t dtype,
                           float ckv_scale, float w_scale, float kv_out_inv_scale,
                           int32_t* d_status, mla_stream_t stream) {
  if (dtype_ok(dtype) && num_heads >= 1 && !c_kv_buf) return MLA_ERR_ARG;
  return upproject_impl(k_nope, v, c_kv_buf, nullptr, nullptr, 0, w_k, w_uv, buffer_lengths, chunk,
                        buffer_token_size, num_heads, dtype, ckv_scale, w_scale, kv_out_inv_scale,
                        d_status, stream);
}

mla_status_t mla_upproject_paged(void* k_nope, void* v, const void* kv_cache,
                                 const int32_t* cache_rows, int32_t num_cache_rows,
                                 const int32_t* buffer_lengths, int32_t chunk,
                                 uint32_t buffer_token_size, const void* w_k, const void* w_uv,
                                 int32_t num_heads, int32_t dtype, float ckv_scale, float w_scale,
                                 float kv_out_inv_scale, int32_t* d_status, mla_stream_t stream) {
  if (dtype_ok(dtype) && num_heads >= 1 && !kv_cache) return MLA_ERR_ARG;
  return upproject_impl(k_nope, v, nullptr, kv_cache, cache_rows, num_cache_rows, w_k, w_uv,
                        buffer_lengths, chunk, buffer_token_size, num_heads, dtype, ckv_scale,
                        w_scale, kv_out_inv_scale, d_status, stream);
}

// k_rope from the [S][64] buffer, or (kv_cache given) from the paged cache.
static mla_status_t attention_impl(void* out, float* lse, float* o_acc, float* lse_acc,
                                   const void* q, const void* k_nope, const void* v,
                                   const void* k_rope, const void* kv_cache,
                                   const int32_t* cache_rows, int32_t num_cache_rows,
                                   const uint32_t* iro,
                                   const uint32_t* cache_lengths, const uint32_t* bro,
                                   const uint32_t* co, const int32_t* bl, int32_t chunk,
                                   int32_t max_chunks, int32_t B, int32_t H,
                                   int32_t max_prompt_len, int32_t T_q, uint32_t S, float scale,
                                   float q_scale, float k_scale, float v_scale, int32_t dtype,
                                   int32_t* d_status, cudaStream_t stream) {
  if (!dtype_ok(dtype)) return MLA_ERR_DTYPE;
  if (H < 1) return MLA_ERR_GEOMETRY;
  if (!out || !q || !k_nope || !v || !iro || !cache_lengths || !bro || !co || !bl ||
      !aligned16(out) || !aligned16(q) || !aligned16(k_nope) || !aligned16(v) || B < 1 ||
      T_q < 0 || max_prompt_len < 0 || chunk < 0 || chunk >= max_chunks || S == 0 ||
      S > 0x7FFFFFFFu)
    return MLA_ERR_ARG;
  if (kv_cache) {
    if (!aligned16(kv_cache) || !cache_rows || num_cache_rows < 1) return MLA_ERR_ARG;
  } else if (!k_rope || !aligned16(k_rope)) {
    return MLA_ERR_ARG;
  }
  if (max_chunks > 1 && (!o_acc || !lse_acc || !aligned16(o_acc))) return MLA_ERR_ARG;
  if (T_q == 0 || max_prompt_len == 0) return MLA_OK;
  AttnArgs a;
  a.out = out;
  a.lse = lse;
  a.o_acc = o_acc;
  a.lse_acc = lse_acc;
  a.q = q;
  a.k_nope = k_nope;
  a.v = v;
  a.k_rope = kv_cache ? nullptr : k_rope;
  a.kv_cache = kv_cache;
  a.cache_rows = cache_rows;
  a.num_cache_rows = num_cache_rows;
  a.iro = iro;
  a.cache_len = cache_lengths;
  a.bro = bro;
  a.co = co;
  a.bl = bl;
  a.chunk = chunk;
  a.max_chunks = max_chunks;
  a.B = B;
  a.H = H;
  a.max_prompt_len = max_prompt_len;
  a.T_q = T_q;
  a.S = S;
  a.scale = scale * q_scale * k_scale;
  a.v_scale = v_scale;
  a.dtype = dtype;
  a.status = d_status;
  return from_cuda(launch_attention(a, stream));
}

mla_status_t mla_prefill_attention(void* out, float* lse, float* o_acc, float* lse_acc,
                                   const void* q, const void* k_nope, const void* v,
                                   const void* k_rope, const uint32_t* input_row_offsets,
                                   const uint32_t* cache_lengths,
                                   const uint32_t* buffer_row_offsets,
                                   const uint32_t* cache_offsets, const int32_t* buffer_lengths,
                                   int32_t chunk, int32_t max_chunks, int32_t batch_size,
                                   int32_t num_heads, int32_t max_prompt_len,
                                   int32_t total_q_tokens, uint32_t buffer_token_size,
                                   float scale, float q_scale, float k_scale, float v_scale,
                                   int32_t dtype, int32_t* d_status, mla_stream_t stream) {
  if (!k_rope) return MLA_ERR_ARG;
  return attention_impl(out, lse, o_acc, lse_acc, q, k_nope, v, k_rope, nullptr, nullptr, 0,
                        input_row_offsets, cache_lengths, buffer_row_offsets, cache_offsets,
                        buffer_lengths, chunk, max_chunks, batch_size, num_heads, max_prompt_len,
                        total_q_tokens, buffer_token_size, scale, q_scale, k_scale, v_scale, dtype,
                        d_status, static_cast<cudaStream_t>(stream));
}

mla_status_t mla_prefill_attention_paged(void* out, float* lse, float* o_acc, float* lse_acc,
                                         const void* q, const void* k_nope, const void* v,
                                         const void* kv_cache, const int32_t* cache_rows,
                                         int32_t num_cache_rows,
                                         const uint32_t* input_row_offsets,
                                         const uint32_t* cache_lengths,
                                         const uint32_t* buffer_row_offsets,
                                         const uint32_t* cache_offsets,
                                         const int32_t* buffer_lengths, int32_t chunk,
                                         int32_t max_chunks, int32_t batch_size,
                                         int32_t num_heads, int32_t max_prompt_len,
                                         int32_t total_q_tokens, uint32_t buffer_token_size,
                                         float scale, float q_scale, float k_scale,
                                         float v_scale, int32_t dtype, int32_t* d_status,
                                         mla_stream_t stream) {
  if (!kv_cache) return MLA_ERR_ARG;
  return attention_impl(out, lse, o_acc, lse_acc, q, k_nope, v, nullptr, kv_cache, cache_rows,
                        num_cache_rows, input_row_offsets, cache_lengths, buffer_row_offsets,
                        cache_offsets, buffer_lengths, chunk, max_chunks, batch_size, num_heads,
                        max_prompt_len, total_q_tokens, buffer_token_size, scale, q_scale, k_scale,
                        v_scale, dtype, d_status, static_cast<cudaStream_t>(stream));
}

size_t mla_prefill_workspace_bytes(int32_t batch_size, int32_t num_heads, int32_t total_q_tokens,
                                   int32_t max_chunks, uint32_t buffer_token_size, int32_t dtype) {
  if (batch_size < 0 || num_heads < 1 || total_q_tokens < 0 || max_chunks < 1 ||
      buffer_token_size == 0 || !dtype_ok(dtype))
    return 0;
  return layout(batch_size, num_heads, total_q_tokens, max_chunks, buffer_token_size, dtype).total;
}

mla_status_t mla_prefill(void* out, float* lse, const void* q, const uint32_t* input_row_offsets,
                         const uint32_t* cache_lengths, const void* kv_cache,
                         const int32_t* page_table, int32_t num_pages, int32_t page_size,
                         int32_t max_pages_per_seq, const void* w_k, const void* w_uv,
                         int32_t batch_size, int32_t num_heads, int32_t total_q_tokens,
                         int32_t max_prompt_len, uint32_t buffer_token_size, int32_t max_chunks,
                         float scale, float q_scale, float ckv_scale, float w_scale,
                         int32_t dtype, void* workspace, size_t workspace_bytes,
                         int32_t* d_status, mla_stream_t stream_) {
  if (!dtype_ok(dtype)) return MLA_ERR_DTYPE;
  if (num_heads < 1) return MLA_ERR_GEOMETRY;
  if (!out || !q || !input_row_offsets || !cache_lengths || !kv_cache || !page_table || !w_k ||
      !w_uv || batch_size < 1 || total_q_tokens < 0 || max_prompt_len < 0 || max_chunks < 1 ||
      buffer_token_size == 0 || buffer_token_size > 0x7FFFFFFFu || num_pages < 1 ||
      page_size < 1 || max_pages_per_seq < 1 || ckv_scale == 0.f || !aligned16(kv_cache) ||
      static_cast<int64_t>(num_pages) * page_size > 0x7FFFFFFFll)
    return MLA_ERR_ARG;
  const Layout L = layout(batch_size, num_heads, total_q_tokens, max_chunks, buffer_token_size, dtype);
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MLA_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* bro = reinterpret_cast<uint32_t*>(ws + L.bro);
  uint32_t* co = reinterpret_cast<uint32_t*>(ws + L.co);
  int32_t* bl = reinterpret_cast<int32_t*>(ws + L.bl);
  float* oacc = max_chunks > 1 ? reinterpret_cast<float*>(ws + L.oacc) : nullptr;
  float* lseacc = max_chunks > 1 ? reinterpret_cast<float*>(ws + L.lseacc) : nullptr;
  if (d_status && cudaMemsetAsync(d_status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return MLA_ERR_LAUNCH;
  mla_status_t st = mla_prefill_plan(bro, co, bl, input_row_offsets, cache_lengths, batch_size,
                                     max_chunks, buffer_token_size, d_status, stream_);
  if (st != MLA_OK) return st;
  // fp8: K and V are stored in the cache's descale domain.
  const float kv_inv = dtype == MLA_E4M3 ? 1.0f / ckv_scale : 1.0f;
  const float kv_descale = dtype == MLA_E4M3 ? ckv_scale : 1.0f;
  // Per chunk: gather the chunk's latent and k_rope rows out of the paged
  // cache, project K_nope / V, attend.  (Reading the rows in place instead,
  // mla_upproject_paged and mla_prefill_attention_paged, measures slower: the
  // projection re-reads every A tile once per head tile, and the copy costs
  // about 1 % of a chunk.)
  for (int c = 0; c < max_chunks; ++c) {
    st = mla_gather_latent(ws + L.ckv, ws + L.krope, kv_cache, page_table, num_pages, page_size,
                           max_pages_per_seq, bro, co, bl, c, batch_size, buffer_token_size,
                           dtype, d_status, stream_);
    if (st != MLA_OK) return st;
    st = mla_upproject(ws + L.knope, ws + L.v, ws + L.ckv, w_k, w_uv, bl, c, buffer_token_size,
                       num_heads, dtype, ckv_scale, w_scale, kv_inv, d_status, stream_);
    if (st != MLA_OK) return st;
    st = attention_impl(out, lse, oacc, lseacc, q, ws + L.knope, ws + L.v, ws + L.krope, nullptr,
                        nullptr, 0, input_row_offsets, cache_lengths, bro, co, bl, c, max_chunks,
                        batch_size, num_heads, max_prompt_len, total_q_tokens, buffer_token_size,
                        scale, q_scale, kv_descale, kv_descale, dtype, d_status, stream);
    if (st != MLA_OK) return st;
  }
  return MLA_OK;
}

int32_t mla_decode_partitions(int32_t batch_size, int32_t num_heads, int32_t max_new_tokens,
                              int32_t max_keys) {
  if (batch_size < 1 || num_heads < 1) return 1;
  return mla::decode_partitioning(batch_size, num_heads, max_new_tokens, max_keys).parts;
}

size_t mla_decode_workspace_bytes(int32_t num_heads, int32_t total_q_tokens, int32_t num_partitions) {
  if (num_heads < 1 || total_q_tokens < 0 || num_partitions < 1) return 0;
  return mla::decode_layout(total_q_tokens, num_heads, num_partitions).total;
}

mla_status_t mla_decode(void* out, float* lse, const void* q, const uint32_t* input_row_offsets,
                        const uint32_t* cache_lengths, const void* kv_cache, const int32_t* page_table,
                        int32_t num_pages, int32_t page_size, int32_t max_pages_per_seq,
                        const void* w_uk, const void* w_uv, int32_t batch_size, int32_t num_heads,
                        int32_t total_q_tokens, int32_t max_new_tokens, int32_t max_seq_len,
                        int32_t num_partitions, float scale, const int32_t* d_indices, int32_t indices_stride,
                        const int32_t* topk_lengths, const float* attn_sink, int32_t dtype,
                        void* workspace, size_t workspace_bytes, int32_t* d_status,
                        mla_stream_t stream) {
  if (dtype != MLA_BF16) return MLA_ERR_DTYPE;
  if (num_heads < 1) return MLA_ERR_GEOMETRY;
  if (!out || !q || !input_row_offsets || !cache_lengths || !kv_cache || !w_uk || !w_uv ||
      !aligned16(out) || !aligned16(q) || !aligned16(kv_cache) || !aligned16(w_uk) ||
      !aligned16(w_uv) || batch_size < 1 || total_q_tokens < 0 || max_new_tokens < 0 ||
      max_seq_len < 1 || num_partitions < 0 || num_pages < 1 || page_size < 1 || !(scale > 0.0f))
    return MLA_ERR_ARG;
  if (d_indices == nullptr && (!page_table || max_pages_per_seq < 1)) return MLA_ERR_ARG;
  if (d_indices != nullptr && indices_stride < 1) return MLA_ERR_ARG;
  const long long rows = static_cast<long long>(total_q_tokens) * num_heads;
  if (rows >= (1ll << 31) / 4 || static_cast<long long>(num_pages) * page_size >= (1ll << 31))
    return MLA_ERR_ARG;
  if (total_q_tokens == 0 || max_new_tokens == 0) return MLA_OK;
  const int max_keys = d_indices != nullptr ? std::min(indices_stride, max_seq_len) : max_seq_len;
  const mla::DecodePartitioning auto_parts =
      mla::decode_partitioning(batch_size, num_heads, max_new_tokens, max_keys);
  const int parts = num_partitions > 0 ? num_partitions : auto_parts.parts;
  const long long items = static_cast<long long>(batch_size) * parts *
                          ((static_cast<long long>(max_new_tokens) * num_heads + 127) / 128);
  if (items >= (1ll << 31)) return MLA_ERR_ARG;
  const mla::DecodeLayout L = mla::decode_layout(total_q_tokens, num_heads, parts);
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MLA_ERR_WORKSPACE;
  mla::DecodeArgs a;
  a.out = out;
  a.lse = lse;
  a.q = q;
  a.kv_cache = kv_cache;
  a.page_table = page_table;
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.max_pages = max_pages_per_seq;
  a.w_uk = w_uk;
  a.w_uv = w_uv;
  a.iro = input_row_offsets;
  a.cache_len = cache_lengths;
  a.B = batch_size;
  a.H = num_heads;
  a.T = total_q_tokens;
  a.max_new = max_new_tokens;
  a.parts = parts;
  a.part_keys = num_partitions > 0 ? 0 : auto_parts.part_keys;
  a.scale = scale;
  a.indices = d_indices;
  a.indices_stride = indices_stride;
  a.topk = topk_lengths;
  a.sink = attn_sink;
  a.workspace = workspace;
  a.status = d_status;
  return from_cuda(mla::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
