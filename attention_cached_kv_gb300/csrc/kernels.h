// kernels.h -- host-side launch interface between the C-ABI layer and the
// kernel translation units.  Host code only; no device code here.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gist_attn.h"

namespace gattn {

// Everything a kernel needs, already validated by the C-ABI layer.
struct Problem {
  const void* q;
  const void* k_new;
  const void* v_new;
  const void* kv_pool;
  const int32_t* item_ids;
  const int32_t* block_table;
  const int32_t* pos_offset;
  void* out;
  int32_t* status;
  int P, l, Hq, Hkv, G, d, block_len, blocks_per_pair, num_blocks, L, layer;
  int C;             // cached keys per pair
  const int32_t* gist_start;  // [P] or nullptr: the gist mask (streaming prefill only)
  int gist_len;
  int flags;                  // GIST_ATTN_FLAG_* (pre-rotated inputs: inv_freq is all 0)
  float scale_log2;  // softmax scale * log2(e)
  float inv_freq[64];  // rope_theta^(-2j/d), j < d/2
  double inv_freq_d[64];  // the same in double (the pool writers rotate in double)
};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// The driver's tensor-map encoder, fetched once through the runtime (no libcuda link).
EncodeTiledFn encode_tiled_fn();

// Each returns GIST_ATTN_OK or a negative GIST_ATTN_ERR_* code.
int launch_prefill(const Problem& pb, cudaStream_t stream);
int launch_prefill_tc(const Problem& pb, cudaStream_t stream);
int launch_prefill_tc_fp8(const Problem& pb, const float* kv_scale, cudaStream_t stream);
int launch_prefill_long(const Problem& pb, cudaStream_t stream);
int launch_prefill_long_on(const Problem& pb, const void* q, const void* k, const void* v, int C,
                           bool f16, const float2* q_base, const float2* q_rel, cudaStream_t stream);
// The staged path (stage.cu): workspace layout, fit and launch (pre-pass + long kernel).
struct StageLayout {
  size_t base_off, rel_off, k_off, v_off, bytes;
};
StageLayout stage_layout(const Problem& pb);
int launch_staged(const Problem& pb, void* workspace, cudaStream_t stream);
int launch_decode(const Problem& pb, cudaStream_t stream);
int launch_decode_long(const Problem& pb, cudaStream_t stream);
int launch_decode_long_fp8(const Problem& pb, const float* kv_scale, cudaStream_t stream);
int launch_decode_short(const Problem& pb, cudaStream_t stream);
int launch_decode_short_fp8(const Problem& pb, const float* kv_scale, cudaStream_t stream);
int launch_gather(const Problem& pb, void* dst, cudaStream_t stream);
int launch_decode_long_stats(const Problem& pb, float* block_mass, cudaStream_t stream);
int launch_decode_gqa(const Problem& pb, cudaStream_t stream);
int launch_decode_gqa_fp8(const Problem& pb, const float* kv_scale, cudaStream_t stream);
int launch_decode_gqa_stats(const Problem& pb, float* block_mass, cudaStream_t stream);
int launch_append(const Problem& pb, void* pool, const int32_t* slot, cudaStream_t stream);
int launch_store(const Problem& pb, void* pool, const int32_t* first_row, const int32_t* store_pos,
                 cudaStream_t stream);
// The projections either side of the attention (gemm.cu).
int launch_qkv_rope(const Problem& pb, const void* x, const void* w, int d_model, void* q,
                    void* kn, void* vn, cudaStream_t stream);
int launch_out_proj(const Problem& pb, const void* attn, const void* w, int d_model, void* y,
                    cudaStream_t stream);

// Whether the prefill kernel can hold this problem's tiles in shared memory.
bool prefill_fits(const Problem& pb);
bool prefill_tc_fits(const Problem& pb);
bool prefill_long_fits(const Problem& pb);
bool prefill_long_grid_ok(const Problem& pb, int rows);
bool staged_fits(const Problem& pb);
bool decode_fits(const Problem& pb);
bool decode_long_fits(const Problem& pb);
bool decode_short_fits(const Problem& pb);
bool decode_long_stats_fits(const Problem& pb);
bool decode_gqa_fits(const Problem& pb);
bool decode_gqa_stats_fits(const Problem& pb);

}  // namespace gattn
