// append.cu -- the two writes into the pool.
//   append: the decode step's new token ([KV page, "Reusable-state"]:
//     K_{<=t} = [K_{<t}; k_t], the new K/V are appended to every layer's cache;
//     [Suffix page, §6 问题四]: the logical slot is found through the block table).
//   store: a compressed item's cache entry ([Gist page, "论文做了什么"]: after
//     the offline pass over [prompt; gist], each layer keeps the K/V at the k
//     gist positions).
// Keys are stored rotated at their positions, in bf16 rounded to nearest even;
// values are copied.  The rotation runs in double: a stored key is read by
// every later step, and an fp32 angle (position x frequency) drifts by about
// position x 2^-24 radians, more than a bf16 step for small rotated values at
// positions in the thousands.  The writes are a few rows per call.
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上";
//        [Suffix page] icman.com.cn news 64898;
//        [KV page] "为什么自回归推理缓存 KV，而不缓存历史 Q？".
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace gattn {
namespace {

// dst[j], dst[j + half] = the pair (src[j], src[j + half]) rotated by `angle`,
// rounded once to bf16 (nearest even) from double.
__device__ __forceinline__ void rotate_pair(const bf16* src, bf16* dst, int j, int half,
                                            double angle) {
  double sn, cs;
  sincos(angle, &sn, &cs);
  const double x = (double)__bfloat162float(src[j]), y = (double)__bfloat162float(src[j + half]);
  dst[j] = __double2bfloat16(x * cs - y * sn);
  dst[j + half] = __double2bfloat16(y * cs + x * sn);
}

struct AppendParams {
  const bf16* k_new;
  const bf16* v_new;
  bf16* pool;
  const int32_t* block_table;
  const int32_t* slot;
  const int32_t* pos_offset;
  int32_t* status;
  int Hkv, d, block_len, blocks_per_pair, num_blocks, L, layer;
  double inv_freq[64];
};

// One warp per (sequence, KV head): lanes take frequency pairs (j, j + d/2).
__global__ void __launch_bounds__(32) append_kernel(const __grid_constant__ AppendParams prm) {
  const int g = blockIdx.x % prm.Hkv, p = blockIdx.x / prm.Hkv, lane = threadIdx.x;
  const int s = prm.slot[p];
  const int C = prm.blocks_per_pair * prm.block_len;
  int32_t blk = -1;
  if (s >= 0 && s < C) blk = prm.block_table[(int64_t)p * prm.blocks_per_pair + s / prm.block_len];
  if (blk < 0 || blk >= prm.num_blocks) {
    if (lane == 0) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
    return;
  }
  const int t = s % prm.block_len, half = prm.d / 2;
  int64_t r = ((int64_t)blk * prm.L + prm.layer) * 2 * prm.Hkv + g;  // K row group
  bf16* krow = prm.pool + (r * prm.block_len + t) * prm.d;
  bf16* vrow = prm.pool + ((r + prm.Hkv) * prm.block_len + t) * prm.d;
  const bf16* k = prm.k_new + ((int64_t)p * prm.Hkv + g) * prm.d;
  const bf16* v = prm.v_new + ((int64_t)p * prm.Hkv + g) * prm.d;
  const double pos = (double)(prm.pos_offset ? prm.pos_offset[p] : s);
  for (int j = lane; j < half; j += 32) rotate_pair(k, krow, j, half, pos * prm.inv_freq[j]);
  for (int e = lane; e < prm.d; e += 32) vrow[e] = v[e];
}

struct StoreParams {
  const bf16* k_new;
  const bf16* v_new;
  bf16* pool;
  const int32_t* item_ids;
  const int32_t* first_row;
  const int32_t* store_pos;
  int32_t* status;
  int l, Hkv, d, k, num_blocks, L, layer;
  double inv_freq[64];
};

// One CTA of 4 warps per (pair, KV head); warps take the k rows in turn, lanes
// the frequency pairs (j, j + d/2) and then the value's elements.
__global__ void __launch_bounds__(128) store_kernel(const __grid_constant__ StoreParams prm) {
  const int g = blockIdx.x % prm.Hkv, p = blockIdx.x / prm.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = prm.first_row[p];
  const int32_t blk = prm.item_ids[p];
  if (r0 < 0 || r0 > prm.l - prm.k || blk < 0 || blk >= prm.num_blocks) {
    if (threadIdx.x == 0) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
    return;
  }
  const int half = prm.d / 2;
  const double pos0 = (double)(prm.store_pos ? prm.store_pos[p] : 0);
  const int64_t r = ((int64_t)blk * prm.L + prm.layer) * 2 * prm.Hkv + g;  // K row group
  for (int t = warp; t < prm.k; t += 4) {
    bf16* krow = prm.pool + (r * prm.k + t) * prm.d;
    bf16* vrow = prm.pool + ((r + prm.Hkv) * prm.k + t) * prm.d;
    const int64_t src = (((int64_t)p * prm.l + r0 + t) * prm.Hkv + g) * prm.d;
    const bf16* k = prm.k_new + src;
    const bf16* v = prm.v_new + src;
    const double pos = pos0 + (double)t;
    for (int j = lane; j < half; j += 32) rotate_pair(k, krow, j, half, pos * prm.inv_freq[j]);
    for (int e = lane; e < prm.d; e += 32) vrow[e] = v[e];
  }
}

}  // namespace

int launch_store(const Problem& pb, void* pool, const int32_t* first_row, const int32_t* store_pos,
                 cudaStream_t stream) {
  StoreParams prm{};
  prm.k_new = static_cast<const bf16*>(pb.k_new);
  prm.v_new = static_cast<const bf16*>(pb.v_new);
  prm.pool = static_cast<bf16*>(pool);
  prm.item_ids = pb.item_ids;
  prm.first_row = first_row;
  prm.store_pos = store_pos;
  prm.status = pb.status;
  prm.l = pb.l;
  prm.Hkv = pb.Hkv;
  prm.d = pb.d;
  prm.k = pb.block_len;
  prm.num_blocks = pb.num_blocks;
  prm.L = pb.L;
  prm.layer = pb.layer;
  for (int j = 0; j < 64; ++j) prm.inv_freq[j] = pb.inv_freq_d[j];
  const int64_t grid = (int64_t)pb.P * pb.Hkv;
  if (grid > 0x7fffffff) return GIST_ATTN_ERR_UNSUPPORTED;
  store_kernel<<<(unsigned)grid, 128, 0, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

int launch_append(const Problem& pb, void* pool, const int32_t* slot, cudaStream_t stream) {
  AppendParams prm{};
  prm.k_new = static_cast<const bf16*>(pb.k_new);
  prm.v_new = static_cast<const bf16*>(pb.v_new);
  prm.pool = static_cast<bf16*>(pool);
  prm.block_table = pb.block_table;
  prm.slot = slot;
  prm.pos_offset = pb.pos_offset;
  prm.status = pb.status;
  prm.Hkv = pb.Hkv;
  prm.d = pb.d;
  prm.block_len = pb.block_len;
  prm.blocks_per_pair = pb.blocks_per_pair;
  prm.num_blocks = pb.num_blocks;
  prm.L = pb.L;
  prm.layer = pb.layer;
  for (int j = 0; j < 64; ++j) prm.inv_freq[j] = pb.inv_freq_d[j];
  const int64_t grid = (int64_t)pb.P * pb.Hkv;
  if (grid > 0x7fffffff) return GIST_ATTN_ERR_UNSUPPORTED;
  append_kernel<<<(unsigned)grid, 32, 0, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

}  // namespace gattn
