// api.cu -- the C ABI declared in include/gist_attn.h: argument checks on the
// host, kernel selection (one route function per entry point, also reported by
// gist_attn_route), and the cache byte-count helpers.
//
// Nothing here allocates device memory or keeps state between calls; the only
// process-wide value is the driver's tensor-map encoder, looked up once.
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上";
//        [KV page] "为什么自回归推理缓存 KV，而不缓存历史 Q？".
#include <math.h>
#include <stdint.h>

#include "gist_attn.h"
#include "kernels.h"

namespace gattn {

EncodeTiledFn encode_tiled_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

namespace {

constexpr int64_t kMaxKeys = 1 << 24;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Checks the dimensions and fills everything of `pb` except the tensor pointers.
int check_dims(const gist_attn_dims* dm, Problem* pb) {
  if (!dm) return GIST_ATTN_ERR_NULL;
  const gist_attn_dims& d = *dm;
  if (d.num_pairs < 0 || d.n_new < 1 || d.num_q_heads < 1 || d.num_kv_heads < 1 ||
      d.num_q_heads % d.num_kv_heads != 0 || d.block_len < 0 || d.blocks_per_pair < 0 ||
      d.num_layers < 1 || d.layer < 0 || d.layer >= d.num_layers || d.num_blocks < 0)
    return GIST_ATTN_ERR_DIMS;
  if (!(d.rope_theta > 0.f) || !isfinite(d.rope_theta) || !(d.softmax_scale >= 0.f) ||
      !isfinite(d.softmax_scale))
    return GIST_ATTN_ERR_DIMS;
  const int64_t C = (int64_t)d.block_len * d.blocks_per_pair;
  if (C + d.n_new > kMaxKeys) return GIST_ATTN_ERR_DIMS;
  if (C > 0 && d.num_blocks < 1) return GIST_ATTN_ERR_DIMS;
  if (d.head_dim != 64 && d.head_dim != 128) return GIST_ATTN_ERR_UNSUPPORTED;
  if (d.num_q_heads / d.num_kv_heads > 256) return GIST_ATTN_ERR_UNSUPPORTED;
  // element counts of the largest arrays must fit comfortably in 64 bits
  const double elems = (double)d.num_pairs * d.n_new * d.num_q_heads * d.head_dim;
  const double pool = (double)d.num_blocks * d.num_layers * 2 * d.num_kv_heads *
                      (double)d.block_len * d.head_dim;
  if (elems > 4e18 || pool > 4e18) return GIST_ATTN_ERR_DIMS;

  pb->status = d.status;
  pb->P = d.num_pairs;
  pb->l = d.n_new;
  pb->Hq = d.num_q_heads;
  pb->Hkv = d.num_kv_heads;
  pb->G = d.num_q_heads / d.num_kv_heads;
  pb->d = d.head_dim;
  pb->block_len = d.block_len;
  pb->blocks_per_pair = d.blocks_per_pair;
  pb->num_blocks = d.num_blocks;
  pb->L = d.num_layers;
  pb->layer = d.layer;
  pb->C = (int)C;
  const double scale = d.softmax_scale > 0.f ? (double)d.softmax_scale : 1.0 / sqrt((double)d.head_dim);
  pb->scale_log2 = (float)(scale * 1.4426950408889634);  // log2(e)
  if (d.flags & ~(GIST_ATTN_FLAG_PREROTATED | GIST_ATTN_FLAG_TEST_WITHHOLD)) return GIST_ATTN_ERR_DIMS;
  // pre-rotated inputs: every rotation angle is 0 (cos 1, sin 0), the identity
  const bool rotate = !(d.flags & GIST_ATTN_FLAG_PREROTATED);
  for (int j = 0; j < 64; ++j) {
    pb->inv_freq_d[j] = rotate && j < d.head_dim / 2
                            ? pow((double)d.rope_theta, -2.0 * j / (double)d.head_dim)
                            : 0.0;
    pb->inv_freq[j] = (float)pb->inv_freq_d[j];
  }
  pb->flags = d.flags;
  return GIST_ATTN_OK;
}

// The cached-segment arguments: pool and exactly one index array when C > 0.
int check_cache_args(const Problem& pb, const void* kv_pool, const int32_t* item_ids,
                     const int32_t* block_table) {
  if (pb.C == 0) return GIST_ATTN_OK;
  if (!kv_pool || (!item_ids && !block_table)) return GIST_ATTN_ERR_NULL;
  if (item_ids && block_table) return GIST_ATTN_ERR_DIMS;
  if (item_ids && pb.blocks_per_pair != 1) return GIST_ATTN_ERR_DIMS;
  if (!aligned(kv_pool, 16) || !aligned(item_ids, 4) || !aligned(block_table, 4))
    return GIST_ATTN_ERR_ALIGN;
  return GIST_ATTN_OK;
}

}  // namespace
}  // namespace gattn

using gattn::Problem;

namespace gattn {
namespace {

// Checks and fills `pb` for gist_attn_fwd / gist_attn_fwd_ws; returns
// GIST_ATTN_OK, or a code to return as is (P == 0 also comes back OK with
// pb->P == 0).
int prepare_fwd(const void* q, const void* k_new, const void* v_new, const void* kv_pool,
                const int32_t* item_ids, const int32_t* block_table, const int32_t* pos_offset,
                void* out, const gist_attn_dims* dims, Problem* pb) {
  int rc = check_dims(dims, pb);
  if (rc != GIST_ATTN_OK || pb->P == 0) return rc;
  if (!q || !k_new || !v_new || !out) return GIST_ATTN_ERR_NULL;
  rc = check_cache_args(*pb, kv_pool, item_ids, block_table);
  if (rc != GIST_ATTN_OK) return rc;
  if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(out, 16) ||
      !aligned(pos_offset, 4) || !aligned(pb->status, 4))
    return GIST_ATTN_ERR_ALIGN;
  pb->q = q;
  pb->k_new = k_new;
  pb->v_new = v_new;
  pb->kv_pool = pb->C > 0 ? kv_pool : nullptr;
  pb->item_ids = pb->C > 0 ? item_ids : nullptr;
  pb->block_table = pb->C > 0 ? block_table : nullptr;
  pb->pos_offset = pos_offset;
  pb->out = out;
  if (pb->C == 0) pb->blocks_per_pair = 0;  // nothing cached: no ids to read
  return GIST_ATTN_OK;
}

// The staged path applies: more than 128 keys on d = 64 where neither
// single-kernel tensor-core path runs.
bool wants_stage(const Problem& pb) {
  return pb.l >= 2 && !prefill_tc_fits(pb) && !prefill_long_fits(pb) && staged_fits(pb);
}

// Kernel selection, one function per entry point: the entry points launch what
// these return, and gist_attn_route reports it.  Each returns a
// GIST_ATTN_ROUTE_* value, or GIST_ATTN_ERR_UNSUPPORTED.

// gist_attn_fwd: the decode kernels for l = 1, then the tensor-core prefill
// (every key of a tile in one pass), the long prefill (pre-rotated, no cache),
// and the streaming prefill for everything else.
int route_fwd(const Problem& pb) {
  if (pb.l == 1) {
    if (decode_long_fits(pb)) return GIST_ATTN_ROUTE_DECODE_LONG;
    if (decode_short_fits(pb)) return GIST_ATTN_ROUTE_DECODE_SHORT;
    if (decode_gqa_fits(pb)) return GIST_ATTN_ROUTE_DECODE_GQA;
    if (decode_fits(pb)) return GIST_ATTN_ROUTE_DECODE;
  }
  if (prefill_tc_fits(pb)) return GIST_ATTN_ROUTE_PREFILL_TC;
  if (prefill_long_fits(pb)) return GIST_ATTN_ROUTE_PREFILL_LONG;
  if (prefill_fits(pb)) return GIST_ATTN_ROUTE_PREFILL_STREAM;
  return GIST_ATTN_ERR_UNSUPPORTED;
}

// gist_attn_fwd_ws with a large enough workspace: the staged path where it
// applies, else as gist_attn_fwd.
int route_fwd_ws(const Problem& pb) {
  return wants_stage(pb) ? GIST_ATTN_ROUTE_STAGED : route_fwd(pb);
}

// gist_attn_fwd_fp8kv: the kernels with an E4M3 variant.
int route_fp8(const Problem& pb) {
  if (prefill_tc_fits(pb)) return GIST_ATTN_ROUTE_PREFILL_TC;
  if (pb.C > 0 && decode_long_fits(pb)) return GIST_ATTN_ROUTE_DECODE_LONG;
  if (decode_short_fits(pb)) return GIST_ATTN_ROUTE_DECODE_SHORT;
  if (decode_gqa_fits(pb)) return GIST_ATTN_ROUTE_DECODE_GQA;
  return GIST_ATTN_ERR_UNSUPPORTED;
}

// gist_attn_fwd_block_mass: the decode kernels with a STATS variant.
int route_block_mass(const Problem& pb) {
  if (pb.C > 0 && decode_long_stats_fits(pb)) return GIST_ATTN_ROUTE_DECODE_LONG;
  if (pb.C > 0 && decode_gqa_stats_fits(pb)) return GIST_ATTN_ROUTE_DECODE_GQA;
  return GIST_ATTN_ERR_UNSUPPORTED;
}

// gist_attn_fwd_gist_mask: the streaming prefill, the one kernel with the mask.
int route_gist_mask(const Problem& pb) {
  return prefill_fits(pb) ? GIST_ATTN_ROUTE_PREFILL_STREAM : GIST_ATTN_ERR_UNSUPPORTED;
}

int dispatch_fwd(const Problem& pb, cudaStream_t stream) {
  switch (route_fwd(pb)) {
    case GIST_ATTN_ROUTE_DECODE_LONG: return launch_decode_long(pb, stream);
    case GIST_ATTN_ROUTE_DECODE_SHORT: return launch_decode_short(pb, stream);
    case GIST_ATTN_ROUTE_DECODE_GQA: return launch_decode_gqa(pb, stream);
    case GIST_ATTN_ROUTE_DECODE: return launch_decode(pb, stream);
    case GIST_ATTN_ROUTE_PREFILL_TC: return launch_prefill_tc(pb, stream);
    case GIST_ATTN_ROUTE_PREFILL_LONG: return launch_prefill_long(pb, stream);
    case GIST_ATTN_ROUTE_PREFILL_STREAM: return launch_prefill(pb, stream);
    default: return GIST_ATTN_ERR_UNSUPPORTED;
  }
}

}  // namespace
}  // namespace gattn

extern "C" int gist_attn_fwd(const void* q, const void* k_new, const void* v_new,
                             const void* kv_pool, const int32_t* item_ids,
                             const int32_t* block_table, const int32_t* pos_offset, void* out,
                             const gist_attn_dims* dims, cudaStream_t stream) {
  Problem pb{};
  const int rc = gattn::prepare_fwd(q, k_new, v_new, kv_pool, item_ids, block_table, pos_offset, out,
                                    dims, &pb);
  if (rc != GIST_ATTN_OK || pb.P == 0) return rc;
  return gattn::dispatch_fwd(pb, stream);
}

extern "C" size_t gist_attn_workspace_bytes(const gist_attn_dims* dims) {
  Problem pb{};
  if (gattn::check_dims(dims, &pb) != GIST_ATTN_OK || pb.P == 0) return 0;
  if (pb.C == 0) pb.blocks_per_pair = 0;
  return gattn::wants_stage(pb) ? gattn::stage_layout(pb).bytes : 0;
}

extern "C" int gist_attn_fwd_ws(const void* q, const void* k_new, const void* v_new,
                                const void* kv_pool, const int32_t* item_ids,
                                const int32_t* block_table, const int32_t* pos_offset, void* out,
                                void* workspace, size_t workspace_bytes,
                                const gist_attn_dims* dims, cudaStream_t stream) {
  Problem pb{};
  const int rc = gattn::prepare_fwd(q, k_new, v_new, kv_pool, item_ids, block_table, pos_offset, out,
                                    dims, &pb);
  if (rc != GIST_ATTN_OK || pb.P == 0) return rc;
  if (workspace && gattn::aligned(workspace, 256) &&
      gattn::route_fwd_ws(pb) == GIST_ATTN_ROUTE_STAGED &&
      workspace_bytes >= gattn::stage_layout(pb).bytes)
    return gattn::launch_staged(pb, workspace, stream);
  return gattn::dispatch_fwd(pb, stream);
}

extern "C" int gist_attn_fwd_fp8kv(const void* q, const void* k_new, const void* v_new,
                                   const void* kv_pool_e4m3, const float* kv_scale,
                                   const int32_t* item_ids, const int32_t* block_table,
                                   const int32_t* pos_offset, void* out,
                                   const gist_attn_dims* dims, cudaStream_t stream) {
  Problem pb{};
  int rc = gattn::check_dims(dims, &pb);
  if (rc != GIST_ATTN_OK) return rc;
  if (pb.P == 0) return GIST_ATTN_OK;
  if (!q || !k_new || !v_new || !out) return GIST_ATTN_ERR_NULL;
  rc = gattn::check_cache_args(pb, kv_pool_e4m3, item_ids, block_table);
  if (rc != GIST_ATTN_OK) return rc;
  if (pb.C > 0 && !kv_scale) return GIST_ATTN_ERR_NULL;
  if (!gattn::aligned(q, 16) || !gattn::aligned(k_new, 16) || !gattn::aligned(v_new, 16) ||
      !gattn::aligned(out, 16) || !gattn::aligned(pos_offset, 4) ||
      !gattn::aligned(pb.status, 4) || !gattn::aligned(kv_scale, 4))
    return GIST_ATTN_ERR_ALIGN;
  pb.q = q;
  pb.k_new = k_new;
  pb.v_new = v_new;
  pb.kv_pool = kv_pool_e4m3;
  pb.item_ids = item_ids;
  pb.block_table = block_table;
  pb.pos_offset = pos_offset;
  pb.out = out;
  switch (gattn::route_fp8(pb)) {
    case GIST_ATTN_ROUTE_PREFILL_TC: return gattn::launch_prefill_tc_fp8(pb, kv_scale, stream);
    case GIST_ATTN_ROUTE_DECODE_LONG: return gattn::launch_decode_long_fp8(pb, kv_scale, stream);
    case GIST_ATTN_ROUTE_DECODE_SHORT: return gattn::launch_decode_short_fp8(pb, kv_scale, stream);
    case GIST_ATTN_ROUTE_DECODE_GQA: return gattn::launch_decode_gqa_fp8(pb, kv_scale, stream);
    default: return GIST_ATTN_ERR_UNSUPPORTED;
  }
}

extern "C" int gist_attn_fwd_block_mass(const void* q, const void* k_new, const void* v_new,
                                        const void* kv_pool, const int32_t* block_table,
                                        const int32_t* pos_offset, void* out, float* block_mass,
                                        const gist_attn_dims* dims, cudaStream_t stream) {
  Problem pb{};
  int rc = gattn::check_dims(dims, &pb);
  if (rc != GIST_ATTN_OK) return rc;
  if (pb.P == 0) return GIST_ATTN_OK;
  if (!q || !k_new || !v_new || !out || !block_mass || !kv_pool || !block_table)
    return GIST_ATTN_ERR_NULL;
  rc = gattn::check_cache_args(pb, kv_pool, nullptr, block_table);
  if (rc != GIST_ATTN_OK) return rc;
  if (!gattn::aligned(q, 16) || !gattn::aligned(k_new, 16) || !gattn::aligned(v_new, 16) ||
      !gattn::aligned(out, 16) || !gattn::aligned(pos_offset, 4) ||
      !gattn::aligned(pb.status, 4) || !gattn::aligned(block_mass, 4))
    return GIST_ATTN_ERR_ALIGN;
  pb.q = q;
  pb.k_new = k_new;
  pb.v_new = v_new;
  pb.kv_pool = kv_pool;
  pb.block_table = block_table;
  pb.pos_offset = pos_offset;
  pb.out = out;
  switch (gattn::route_block_mass(pb)) {
    case GIST_ATTN_ROUTE_DECODE_LONG: return gattn::launch_decode_long_stats(pb, block_mass, stream);
    case GIST_ATTN_ROUTE_DECODE_GQA: return gattn::launch_decode_gqa_stats(pb, block_mass, stream);
    default: return GIST_ATTN_ERR_UNSUPPORTED;
  }
}

extern "C" int gist_kv_append(const void* k_new, const void* v_new, void* kv_pool,
                              const int32_t* block_table, const int32_t* slot,
                              const int32_t* pos_offset, const gist_attn_dims* dims,
                              cudaStream_t stream) {
  Problem pb{};
  int rc = gattn::check_dims(dims, &pb);
  if (rc != GIST_ATTN_OK) return rc;
  if (pb.P == 0) return GIST_ATTN_OK;
  if (pb.l != 1 || pb.C == 0) return GIST_ATTN_ERR_DIMS;
  if (!k_new || !v_new || !kv_pool || !block_table || !slot) return GIST_ATTN_ERR_NULL;
  if (!gattn::aligned(k_new, 16) || !gattn::aligned(v_new, 16) || !gattn::aligned(kv_pool, 16) ||
      !gattn::aligned(block_table, 4) || !gattn::aligned(slot, 4) ||
      !gattn::aligned(pos_offset, 4) || !gattn::aligned(pb.status, 4))
    return GIST_ATTN_ERR_ALIGN;
  pb.k_new = k_new;
  pb.v_new = v_new;
  pb.block_table = block_table;
  pb.pos_offset = pos_offset;
  return gattn::launch_append(pb, kv_pool, slot, stream);
}

extern "C" int gist_attn_fwd_gist_mask(const void* q, const void* k_new, const void* v_new,
                                       const void* kv_pool, const int32_t* item_ids,
                                       const int32_t* block_table, const int32_t* pos_offset,
                                       const int32_t* gist_start, int gist_len, void* out,
                                       const gist_attn_dims* dims, cudaStream_t stream) {
  Problem pb{};
  int rc = gattn::check_dims(dims, &pb);
  if (rc != GIST_ATTN_OK) return rc;
  if (gist_len < 0) return GIST_ATTN_ERR_DIMS;
  if (pb.P == 0) return GIST_ATTN_OK;
  if (!q || !k_new || !v_new || !out || !gist_start) return GIST_ATTN_ERR_NULL;
  rc = gattn::check_cache_args(pb, kv_pool, item_ids, block_table);
  if (rc != GIST_ATTN_OK) return rc;
  if (!gattn::aligned(q, 16) || !gattn::aligned(k_new, 16) || !gattn::aligned(v_new, 16) ||
      !gattn::aligned(out, 16) || !gattn::aligned(pos_offset, 4) ||
      !gattn::aligned(gist_start, 4) || !gattn::aligned(pb.status, 4))
    return GIST_ATTN_ERR_ALIGN;
  pb.q = q;
  pb.k_new = k_new;
  pb.v_new = v_new;
  pb.kv_pool = pb.C > 0 ? kv_pool : nullptr;
  pb.item_ids = pb.C > 0 ? item_ids : nullptr;
  pb.block_table = pb.C > 0 ? block_table : nullptr;
  pb.pos_offset = pos_offset;
  pb.out = out;
  pb.gist_start = gist_start;
  pb.gist_len = gist_len;
  if (pb.C == 0) pb.blocks_per_pair = 0;
  if (gattn::route_gist_mask(pb) != GIST_ATTN_ROUTE_PREFILL_STREAM) return GIST_ATTN_ERR_UNSUPPORTED;
  return gattn::launch_prefill(pb, stream);
}

extern "C" int gist_kv_store(const void* k_new, const void* v_new, void* kv_pool,
                             const int32_t* item_ids, const int32_t* first_row,
                             const int32_t* store_pos, const gist_attn_dims* dims,
                             cudaStream_t stream) {
  Problem pb{};
  int rc = gattn::check_dims(dims, &pb);
  if (rc != GIST_ATTN_OK) return rc;
  if (pb.P == 0) return GIST_ATTN_OK;
  if (pb.blocks_per_pair != 1 || pb.block_len < 1 || pb.block_len > pb.l)
    return GIST_ATTN_ERR_DIMS;
  if (!k_new || !v_new || !kv_pool || !item_ids || !first_row) return GIST_ATTN_ERR_NULL;
  if (!gattn::aligned(k_new, 16) || !gattn::aligned(v_new, 16) || !gattn::aligned(kv_pool, 16) ||
      !gattn::aligned(item_ids, 4) || !gattn::aligned(first_row, 4) ||
      !gattn::aligned(store_pos, 4) || !gattn::aligned(pb.status, 4))
    return GIST_ATTN_ERR_ALIGN;
  pb.k_new = k_new;
  pb.v_new = v_new;
  pb.item_ids = item_ids;
  return gattn::launch_store(pb, kv_pool, first_row, store_pos, stream);
}

extern "C" int gist_qkv_rope(const void* x, const void* w_qkv, const int32_t* pos_offset, void* q,
                             void* k_new, void* v_new, int d_model, const gist_attn_dims* dims,
                             cudaStream_t stream) {
  Problem pb{};
  if (dims && (dims->flags & GIST_ATTN_FLAG_PREROTATED)) return GIST_ATTN_ERR_DIMS;
  int rc = gattn::check_dims(dims, &pb);
  if (rc != GIST_ATTN_OK) return rc;
  if (d_model < 1) return GIST_ATTN_ERR_DIMS;
  if (pb.P == 0) return GIST_ATTN_OK;
  if (!x || !w_qkv || !q || !k_new || !v_new) return GIST_ATTN_ERR_NULL;
  if (!gattn::aligned(x, 16) || !gattn::aligned(w_qkv, 16) || !gattn::aligned(q, 16) ||
      !gattn::aligned(k_new, 16) || !gattn::aligned(v_new, 16) || !gattn::aligned(pos_offset, 4) ||
      !gattn::aligned(pb.status, 4))
    return GIST_ATTN_ERR_ALIGN;
  pb.pos_offset = pos_offset;
  return gattn::launch_qkv_rope(pb, x, w_qkv, d_model, q, k_new, v_new, stream);
}

extern "C" int gist_out_proj(const void* attn_out, const void* w_o, void* y, int d_model,
                             const gist_attn_dims* dims, cudaStream_t stream) {
  Problem pb{};
  int rc = gattn::check_dims(dims, &pb);
  if (rc != GIST_ATTN_OK) return rc;
  if (d_model < 1) return GIST_ATTN_ERR_DIMS;
  if (pb.P == 0) return GIST_ATTN_OK;
  if (!attn_out || !w_o || !y) return GIST_ATTN_ERR_NULL;
  if (!gattn::aligned(attn_out, 16) || !gattn::aligned(w_o, 16) || !gattn::aligned(y, 16) ||
      !gattn::aligned(pb.status, 4))
    return GIST_ATTN_ERR_ALIGN;
  return gattn::launch_out_proj(pb, attn_out, w_o, d_model, y, stream);
}

extern "C" int gist_attn_gather_debug(const void* kv_pool, const int32_t* item_ids,
                                      const int32_t* block_table, void* dst,
                                      const gist_attn_dims* dims, cudaStream_t stream) {
  Problem pb{};
  int rc = gattn::check_dims(dims, &pb);
  if (rc != GIST_ATTN_OK) return rc;
  if (pb.P == 0 || pb.C == 0) return GIST_ATTN_OK;
  if (!dst) return GIST_ATTN_ERR_NULL;
  rc = gattn::check_cache_args(pb, kv_pool, item_ids, block_table);
  if (rc != GIST_ATTN_OK) return rc;
  if (!gattn::aligned(dst, 16) || !gattn::aligned(pb.status, 4)) return GIST_ATTN_ERR_ALIGN;
  pb.kv_pool = kv_pool;
  pb.item_ids = item_ids;
  pb.block_table = block_table;
  return gattn::launch_gather(pb, dst, stream);
}

extern "C" size_t gist_kv_bytes_per_position(int L, int Hkv, int d, int elem_bytes) {
  if (L < 0 || Hkv < 0 || d < 0 || elem_bytes < 0) return 0;
  return (size_t)2 * L * Hkv * d * elem_bytes;
}

extern "C" size_t gist_kv_bytes_per_item(int L, int Hkv, int d, int k, int elem_bytes) {
  if (k < 0) return 0;
  return (size_t)k * gist_kv_bytes_per_position(L, Hkv, d, elem_bytes);
}

extern "C" size_t gist_kv_bytes_batch(int B, int L, int T, int Hkv, int d, int elem_bytes) {
  if (B < 0 || T < 0) return 0;
  return (size_t)B * T * gist_kv_bytes_per_position(L, Hkv, d, elem_bytes);
}

extern "C" int gist_attn_route(int entry, const gist_attn_dims* dims) {
  Problem pb{};
  const int rc = gattn::check_dims(dims, &pb);
  if (rc != GIST_ATTN_OK) return rc;
  if (pb.P == 0) return GIST_ATTN_ROUTE_NONE;
  switch (entry) {
    case GIST_ATTN_ENTRY_FWD:
    case GIST_ATTN_ENTRY_FWD_WS:
      if (pb.C == 0) pb.blocks_per_pair = 0;  // as prepare_fwd leaves it
      return entry == GIST_ATTN_ENTRY_FWD ? gattn::route_fwd(pb) : gattn::route_fwd_ws(pb);
    case GIST_ATTN_ENTRY_FP8KV: return gattn::route_fp8(pb);
    case GIST_ATTN_ENTRY_BLOCK_MASS: return gattn::route_block_mass(pb);
    case GIST_ATTN_ENTRY_GIST_MASK:
      if (pb.C == 0) pb.blocks_per_pair = 0;
      return gattn::route_gist_mask(pb);
    default: return GIST_ATTN_ERR_UNSUPPORTED;
  }
}

extern "C" const char* gist_attn_status_string(int status) {
  switch (status) {
    case GIST_ATTN_OK: return "ok";
    case GIST_ATTN_ERR_NULL: return "a required pointer is NULL";
    case GIST_ATTN_ERR_DIMS: return "inconsistent or out-of-range dimensions";
    case GIST_ATTN_ERR_UNSUPPORTED: return "unsupported head_dim, group size or problem size";
    case GIST_ATTN_ERR_ALIGN: return "a pointer is not aligned as required";
    case GIST_ATTN_ERR_LAUNCH: return "the CUDA launch failed";
    case GIST_ATTN_ERR_SCRATCH:
      return "the call needs more scratch than the library's fixed no-allocation array holds";
    case GIST_ATTN_STATUS_BAD_BLOCK: return "device: a block id was out of range (pair zeroed)";
    case GIST_ATTN_STATUS_TIMEOUT: return "device: a bounded wait on an asynchronous copy gave up";
    case GIST_ATTN_STATUS_BAD_BLOCK | GIST_ATTN_STATUS_TIMEOUT:
      return "device: out-of-range block id and a timed-out wait";
    case GIST_ATTN_STATUS_RANGE:
      return "device: a softmax row was not finite in fp32 (a NaN input or values near the fp32 limit)";
    default: return status < 0 ? "unknown error" : "unknown device status bits";
  }
}
