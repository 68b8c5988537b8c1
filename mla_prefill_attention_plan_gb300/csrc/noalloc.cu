// Prefill attention with the cross-chunk merge state held in a fixed array
// inside this library, for callers that cannot allocate device memory.
//
// Who needs this: code that runs where some other component owns every byte of
// device memory and gives the caller no allocator (a custom operator loaded
// into a serving engine's private memory pool, for instance), and loops that
// must not call cudaMalloc because it synchronises the whole device.  Such a
// caller can pass its inputs and outputs but has nowhere to put the fp32
// O / LSE scratch that mla_prefill_attention needs when a plan has more than
// one chunk.  This entry point uses a statically sized device array instead.
//
// The array lives in this library's device image, so every GPU that loads the
// library holds it (MLA_NOALLOC_MAX_ROWS * 129 floats, about 16.9 MB) until the
// process exits.  Host code never uses the array's name as an address: every
// call looks up the array's device address on the current device with
// cudaGetSymbolAddress and passes that to the kernel.  (Looking it up on every
// call, rather than once per device, keeps the address right after a
// cudaDeviceReset or a reload of the module; the lookup is a host-side table
// read once the module is loaded.)
#include "kernels.cuh"

namespace {

constexpr size_t kMaxRows = MLA_NOALLOC_MAX_ROWS;  // total_q_tokens * num_heads

// [kMaxRows][128] running O, then [kMaxRows] running LSE, all fp32.
static __device__ __align__(256) float g_merge_scratch[kMaxRows * 128 + kMaxRows];

// Device address of the scratch on the current device; null on failure.
float* scratch_on_current_device() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_merge_scratch) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<float*>(ptr);
}

}  // namespace

extern "C" mla_status_t mla_prefill_attention_noalloc(
    void* out, float* lse, const void* q, const void* k_nope, const void* v, const void* k_rope,
    const uint32_t* input_row_offsets, const uint32_t* cache_lengths,
    const uint32_t* buffer_row_offsets, const uint32_t* cache_offsets,
    const int32_t* buffer_lengths, int32_t chunk, int32_t max_chunks, int32_t batch_size,
    int32_t num_heads, int32_t max_prompt_len, int32_t total_q_tokens,
    uint32_t buffer_token_size, float scale, float q_scale, float k_scale, float v_scale,
    int32_t dtype, int32_t* d_status, mla_stream_t stream) {
  if (num_heads < 1 || total_q_tokens < 0) return MLA_ERR_ARG;
  if (static_cast<size_t>(total_q_tokens) * static_cast<size_t>(num_heads) > kMaxRows)
    return MLA_ERR_WORKSPACE;  // beyond the fixed scratch: use mla_prefill_attention
  float* base = scratch_on_current_device();
  if (base == nullptr) return MLA_ERR_LAUNCH;
  // No part of the scratch needs clearing: the first chunk that holds a row's
  // keys writes that row's O and LSE before any later chunk reads them.
  float* o_acc = base;
  float* lse_acc = base + kMaxRows * 128;
  return mla_prefill_attention(out, lse, o_acc, lse_acc, q, k_nope, v, k_rope, input_row_offsets,
                               cache_lengths, buffer_row_offsets, cache_offsets, buffer_lengths,
                               chunk, max_chunks, batch_size, num_heads, max_prompt_len,
                               total_q_tokens, buffer_token_size, scale, q_scale, k_scale, v_scale,
                               dtype, d_status, stream);
}
