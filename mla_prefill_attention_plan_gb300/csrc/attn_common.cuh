// Pieces shared by the attention kernels: launch parameters, the work item of
// one (sequence, 128-query tile, head), and the epilogue of one query row
// (normalisation, natural-log LSE, merge with earlier chunks, bf16 store).
#pragma once
#include "kernels.cuh"

namespace mla {
namespace {

constexpr int BM = 128, BN = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kNegInf = -__builtin_huge_valf();

struct Params {
  __nv_bfloat16* out;
  float* lse;
  float* o_acc;
  float* lse_acc;
  const uint32_t* iro;
  const uint32_t* cache_len;
  const uint32_t* bro;
  const uint32_t* co;
  const int32_t* bl;
  int chunk, B, H, n_qtiles, head_group;
  int T_q;            // rows of q / out / lse: no query row at or past it is read or written
  float scale_log2;   // softmax scale * descales * log2(e)
  float v_scale;
  int32_t* status;
};

// k_rope straight from the paged cache (the PAGED kernels, a launch
// parameter of its own): buffer row r is cache row cache_rows[r]
// (< num_cache_rows, each cache_row_bytes long).
struct PagedRope {
  const uint8_t* kv_cache;
  const int32_t* cache_rows;
  int num_cache_rows, cache_row_bytes;
};

// One work item, as every role sees it.
struct Item {
  int b, h;
  int i0;        // first query row (within the sequence) of the tile
  int nq;        // valid query rows in the tile
  int q_row0;    // first query row in q / out
  int kv_row0;   // first buffer row of the sequence's keys in this chunk
  int n_cb;      // keys of the sequence in this chunk
  int co;        // context position of the first of those keys
  int cb;        // cached tokens of the sequence
  int n_kv;      // 128-key tiles to visit (0: nothing to do)
};

// The work item of query tile `qt` of sequence `b` and head `h` in this
// chunk; false when the tile has no query rows or sees none of the chunk's keys.
__device__ __forceinline__ bool tile_item(const Params& p, int b, int h, int qt, Item& it) {
  it.b = b;
  it.h = h;
  // Every table read first: they are independent, so they share one round
  // trip to L2 (the tables are read-only while the kernel runs).
  const uint32_t* bro_c = p.bro + static_cast<size_t>(p.chunk) * (p.B + 1);
  const uint32_t r0u = __ldg(bro_c + b), r1u = __ldg(bro_c + b + 1);
  const uint32_t qa = __ldg(p.iro + b), qe = __ldg(p.iro + b + 1);
  const uint32_t cou = __ldg(p.co + static_cast<size_t>(p.chunk) * p.B + b);
  const uint32_t cbu = __ldg(p.cache_len + b);
  const int r0 = static_cast<int>(r0u);
  it.n_cb = static_cast<int>(r1u) - r0;
  it.i0 = qt * BM;
  it.n_kv = 0;
  if (qe > static_cast<uint32_t>(p.T_q)) {
    // Offsets past the q / out rows: report them and leave the sequence out
    // (a decreasing pair is simply empty).
    set_status(p.status, MLA_DEV_BAD_OFFSETS);
    it.nq = 0;
    return false;
  }
  const int q0 = static_cast<int>(qa);
  const int new_b = qe >= qa ? static_cast<int>(qe - qa) : 0;
  it.nq = max(0, min(BM, new_b - it.i0));
  it.q_row0 = q0 + it.i0;
  it.kv_row0 = r0;
  it.co = static_cast<int>(cou);
  it.cb = static_cast<int>(cbu);
  if (it.n_cb <= 0 || it.nq <= 0) return false;
  // Keys visible to the tile's last row: relative key index <= last.
  const long long last = static_cast<long long>(it.cb) + it.i0 + it.nq - 1 - it.co;
  if (last < 0) return false;
  const long long nkeys = min(static_cast<long long>(it.n_cb), last + 1);
  it.n_kv = static_cast<int>((nkeys + BN - 1) / BN);
  return true;
}

// The table entry of the item's key `k` (0-based within the sequence's keys
// in this chunk), or 0 past them: a plain load, checked where it is used
// (checked_cache_row), so that it can be issued a stage ahead.
__device__ __forceinline__ int cache_row_entry(const PagedRope& pr, const Item& it, int k) {
  return k < it.n_cb ? __ldg(pr.cache_rows + it.kv_row0 + k) : 0;
}
// A table entry outside the cache is reported and read as row 0 (that key's
// score is then meaningless).
__device__ __forceinline__ int checked_cache_row(const Params& p, const PagedRope& pr, int row) {
  if (static_cast<unsigned>(row) < static_cast<unsigned>(pr.num_cache_rows)) return row;
  set_status(p.status, MLA_DEV_BAD_PAGE);
  return 0;
}

// Epilogue of one query row: O / l, this chunk's natural-log LSE, merge with
// the running result of earlier chunks, then either the final bf16 row (the
// chunk that holds the row's own position) or the fp32 running state.
__device__ __forceinline__ void store_row(const Params& p, const Item& cur, int row, long long qpos,
                                          float m_run, float l_run, const float (&o)[128]) {
  if (row >= cur.nq || qpos < cur.co) return;   // padding row, or finished in an earlier chunk
  const bool first = cur.co == 0;
  const bool final_chunk = qpos < static_cast<long long>(cur.co) + cur.n_cb;
  // Without merge scratch (a one-chunk call) a row can only be finished here;
  // anything else means the plan overflowed max_chunks.
  if ((!first || !final_chunk) && (p.o_acc == nullptr || p.lse_acc == nullptr)) {
    set_status(p.status, MLA_DEV_TOO_MANY_CHUNKS);
    return;
  }
  const size_t t = static_cast<size_t>(cur.q_row0 + row);
  const size_t th = t * p.H + cur.h;
  const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
  const float lse_c = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : kNegInf;
  float w_c = inv;     // weight of this chunk's unnormalised O
  float w_a = 0.f;     // weight of the running result
  float lse_tot = lse_c;
  if (!first) {
    const float lse_a = p.lse_acc[th];
    const float mm = fmaxf(lse_a, lse_c);
    const float ea = __expf(lse_a - mm), ec = __expf(lse_c - mm);
    const float tot = ea + ec;
    w_a = ea / tot;
    w_c = inv * (ec / tot);
    lse_tot = mm + __logf(tot);
  }
  const float4* oa = first ? nullptr : reinterpret_cast<const float4*>(p.o_acc + th * 128);
  if (final_chunk) {
    uint4* dst = reinterpret_cast<uint4*>(p.out + th * 128);
    const float vs = p.v_scale;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) y[i] = o[c * 8 + i] * w_c;
      if (!first) {
        const float4 a0 = oa[2 * c], a1 = oa[2 * c + 1];
        y[0] += w_a * a0.x; y[1] += w_a * a0.y; y[2] += w_a * a0.z; y[3] += w_a * a0.w;
        y[4] += w_a * a1.x; y[5] += w_a * a1.y; y[6] += w_a * a1.z; y[7] += w_a * a1.w;
      }
      dst[c] = make_uint4(pack_bf16(y[0] * vs, y[1] * vs), pack_bf16(y[2] * vs, y[3] * vs),
                          pack_bf16(y[4] * vs, y[5] * vs), pack_bf16(y[6] * vs, y[7] * vs));
    }
    if (p.lse) p.lse[th] = lse_tot;
  } else {
    float4* dst = reinterpret_cast<float4*>(p.o_acc + th * 128);
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      float4 y = make_float4(o[4 * c] * w_c, o[4 * c + 1] * w_c, o[4 * c + 2] * w_c, o[4 * c + 3] * w_c);
      if (!first) {
        const float4 a = oa[c];
        y.x += w_a * a.x; y.y += w_a * a.y; y.z += w_a * a.z; y.w += w_a * a.w;
      }
      dst[c] = y;
    }
    p.lse_acc[th] = lse_tot;
  }
}

}  // namespace
}  // namespace mla
