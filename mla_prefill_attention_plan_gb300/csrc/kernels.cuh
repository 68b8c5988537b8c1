// Internal launchers of the sm_103a kernels (host side).  The public C ABI in
// mla_prefill.h validates arguments and calls these.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm100.cuh"

namespace mla {

// Launch with programmatic stream serialization: the kernel may begin while
// the previous kernel of the stream finishes; it calls pdl_enter() before it
// touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

cudaError_t launch_plan(uint32_t* bro, uint32_t* co, int32_t* bl, const uint32_t* iro,
                        const uint32_t* cache_len, int B, int max_chunks, uint32_t S,
                        int32_t* status, cudaStream_t stream);

struct CacheWriteArgs {
  void* kv_cache;
  void* q;                  // bf16 [T][H][192] or null
  const void* kv_latent;    // bf16 [T][576]
  const float* gamma;       // [512]
  const float* freqs;       // [max_seq_len][64]
  const uint32_t* iro;
  const uint32_t* cache_len;
  const int32_t* page_table;
  int num_pages, page_size, max_pages, B, H, T, max_seq_len;
  float eps, inv_scale;
  int elt_bytes;            // cache storage: 2 (bf16) or 1 (e4m3)
  int32_t* status;
};
cudaError_t launch_cache_write(const CacheWriteArgs& a, cudaStream_t stream);

cudaError_t launch_gather(void* c_kv_buf, void* k_rope_buf, const void* kv_cache,
                          const int32_t* page_table, int num_pages, int page_size, int max_pages,
                          const uint32_t* bro, const uint32_t* co, const int32_t* bl, int chunk,
                          int B, uint32_t S, int elt_bytes, int32_t* status, cudaStream_t stream);

// Per chunk, the cache row of every buffer row (gather.cu).
cudaError_t launch_cache_rows(int32_t* cache_rows, const int32_t* page_table, int num_pages,
                              int page_size, int max_pages, const uint32_t* bro, const uint32_t* co,
                              const int32_t* bl, int max_chunks, int B, uint32_t S, int32_t* status,
                              cudaStream_t stream);

struct UpprojArgs {
  void* k_nope;
  void* v;
  const void* c_kv;
  const void* w_k;
  const void* w_uv;
  const int32_t* buffer_lengths;
  int chunk;
  uint32_t S;
  int H;
  int dtype;
  float out_scale;
  int32_t* status;
  // A rows straight from the paged cache (kv_cache given): buffer row r of
  // the chunk is cache row cache_rows[r] (< num_cache_rows).
  const void* kv_cache = nullptr;
  const int32_t* cache_rows = nullptr;
  int num_cache_rows = 0;
};
// The GEMM on two-SM pairs (cta_group::2 clusters, 256 x 256 tiles); an
// error where the device cannot keep such a cluster resident.
cudaError_t launch_upproject(const UpprojArgs& a, cudaStream_t stream);

struct AttnArgs {
  void* out;
  float* lse;
  float* o_acc;
  float* lse_acc;
  const void* q;
  const void* k_nope;
  const void* v;
  const void* k_rope;           // [S][64] buffer, or null when k_rope comes from the paged cache
  const void* kv_cache = nullptr;      // paged cache rows [num_cache_rows][576] (k_rope = columns 512..575)
  const int32_t* cache_rows = nullptr;  // the chunk's cache row of each buffer row
  int num_cache_rows = 0;
  const uint32_t* iro;
  const uint32_t* cache_len;
  const uint32_t* bro;
  const uint32_t* co;
  const int32_t* bl;
  int chunk;
  int max_chunks;
  int B;
  int H;
  int max_prompt_len;
  int T_q;
  uint32_t S;
  float scale;  // softmax scale times the q and k descales
  float v_scale;
  int dtype;
  int32_t* status;
};
// bf16 attention on two-SM pairs (cta_group::2 clusters); e4m3 Q / K with V
// as f16 holding e4m3-rounded values (as mla_upproject writes it), on the
// same pairs.  An error where the device cannot keep such a cluster resident.
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_attention_pair(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_attention_pair_e4m3(const AttnArgs& a, cudaStream_t stream);

// Absorbed MLA decode (decode.cu).
struct DecodeArgs {
  void* out;                  // [T][H][128] bf16
  float* lse;                 // [T][H] or null
  const void* q;              // [T][H][192] bf16
  const void* kv_cache;       // [num_pages][page_size][576] bf16
  const int32_t* page_table;  // [B][max_pages]
  int num_pages = 0, page_size = 0, max_pages = 0;
  const void* w_uk;           // [H][512][128] bf16
  const void* w_uv;           // [H][128][512] bf16
  const uint32_t* iro;
  const uint32_t* cache_len;
  int B, H, T, max_new, parts;
  int part_keys;              // > 0: about this many keys a partition, at most `parts` of them
  float scale;
  const int32_t* indices;     // sparse: [B][indices_stride] physical cache rows, or null
  int indices_stride;
  const int32_t* topk;        // sparse: [B] or null
  const float* sink;          // [B] or null
  void* workspace;
  int32_t* status;
};
struct DecodeLayout {
  size_t q_full, o_part, lse_part, o_lat, total;
};
DecodeLayout decode_layout(int T, int H, int parts);
// The library's partitioning: about part_keys keys a partition (at most
// `parts` of them), from the batch's sizes and its longest key list.
constexpr int kDecodeMaxParts = 64;
struct DecodePartitioning {
  int parts, part_keys;
};
DecodePartitioning decode_partitioning(int B, int H, int max_new, int max_keys);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// Self-test of the bounded waits (selftest.cu): one cluster of `cluster`
// CTAs waiting on barriers nothing arrives at.
cudaError_t launch_bounded_wait_selftest(int32_t* status, long long* elapsed_ns, uint64_t limit_ns,
                                         int cluster, cudaStream_t stream);

// Tensor-map encoder and device properties (abi.cu).
bool encode_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, uint64_t inner,
               uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle);
int sm_count();

}  // namespace mla
