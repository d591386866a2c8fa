// append.cu -- the decode step's write of the new token's K/V into the paged
// cache ([KV page, "Reusable-state"]: K_{<=t} = [K_{<t}; k_t], the new K/V
// are appended to every layer's cache; [Suffix page, §6 问题四]: the logical
// slot is found through the block table).  The key is stored rotated at its
// position, in bf16 rounded to nearest even; the value is copied.
//
// Pages: [Suffix page] icman.com.cn news 64898;
//        [KV page] "为什么自回归推理缓存 KV，而不缓存历史 Q？".
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace gattn {
namespace {

struct AppendParams {
  const bf16* k_new;
  const bf16* v_new;
  bf16* pool;
  const int32_t* block_table;
  const int32_t* slot;
  const int32_t* pos_offset;
  int32_t* status;
  int Hkv, d, block_len, blocks_per_pair, num_blocks, L, layer;
  float inv_freq[64];
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
  const float pos = (float)(prm.pos_offset ? prm.pos_offset[p] : s);
  for (int j = lane; j < half; j += 32) {
    float sn, cs;
    sincosf(pos * prm.inv_freq[j], &sn, &cs);
    const float x = __bfloat162float(k[j]), y = __bfloat162float(k[j + half]);
    krow[j] = __float2bfloat16_rn(x * cs - y * sn);
    krow[j + half] = __float2bfloat16_rn(y * cs + x * sn);
  }
  for (int e = lane; e < prm.d; e += 32) vrow[e] = v[e];
}

}  // namespace

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
  for (int j = 0; j < 64; ++j) prm.inv_freq[j] = pb.inv_freq[j];
  const int64_t grid = (int64_t)pb.P * pb.Hkv;
  if (grid > 0x7fffffff) return GIST_ATTN_ERR_UNSUPPORTED;
  append_kernel<<<(unsigned)grid, 32, 0, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

}  // namespace gattn
