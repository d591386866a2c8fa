// gather.cu -- writes out, bit for bit, the cached rows each pair reads.
//
// It resolves block ids and addresses with the same pool_block_id / pool_row
// routines the attention kernels use ([Gist page, "在线的一次 attention"]:
// cache[item].K[layer] and .V[layer]; [Suffix page, §6 问题四]: logical block
// -> physical block through an index table), so the test that compares its
// output with a host-side gather checks the attention kernels' addressing.
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上";
//        [Suffix page] icman.com.cn news 64898.
#include "common.cuh"
#include "kernels.h"

namespace gattn {
namespace {

constexpr int kThreads = 256;

// One CTA per (pair, KV head, K or V); dst[p][g][kv][C][d].
__global__ void __launch_bounds__(kThreads) gather_kernel(PoolView pv, bf16* dst, int C, int32_t* status) {
  const int kv = blockIdx.x & 1;
  const int g = (blockIdx.x >> 1) % pv.num_kv_heads;
  const int p = (blockIdx.x >> 1) / pv.num_kv_heads;
  const int cpr = pv.head_dim / 8;
  bf16* out = dst + ((((int64_t)p * pv.num_kv_heads + g) * 2 + kv) * C) * pv.head_dim;

  bool bad = false;
  for (int b = 0; b < pv.blocks_per_pair; ++b) bad |= !pool_block_ok(pv, pool_block_id(pv, p, b));
  if (bad) {
    for (int idx = threadIdx.x; idx < C * cpr; idx += kThreads)
      *reinterpret_cast<uint4*>(out + (int64_t)idx * 8) = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) report(status, GIST_ATTN_STATUS_BAD_BLOCK);
    return;
  }
  for (int idx = threadIdx.x; idx < C * cpr; idx += kThreads) {
    const int kappa = idx / cpr, c = idx - kappa * cpr;
    const int b = kappa / pv.block_len;
    const bf16* src = pool_row(pv, pool_block_id(pv, p, b), g, kv, kappa - b * pv.block_len) + c * 8;
    *reinterpret_cast<uint4*>(out + (int64_t)kappa * pv.head_dim + c * 8) = ldg16(src);
  }
}

}  // namespace

int launch_gather(const Problem& pb, void* dst, cudaStream_t stream) {
  const int64_t grid = (int64_t)pb.P * pb.Hkv * 2;
  if (grid > 0x7fffffff) return GIST_ATTN_ERR_UNSUPPORTED;
  if (grid == 0 || pb.C == 0) return GIST_ATTN_OK;
  PoolView pv{static_cast<const bf16*>(pb.kv_pool), pb.item_ids, pb.block_table, pb.blocks_per_pair,
              pb.block_len, pb.num_blocks, pb.L, pb.layer, pb.Hkv, pb.d};
  gather_kernel<<<(unsigned)grid, kThreads, 0, stream>>>(pv, static_cast<bf16*>(dst), pb.C, pb.status);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

}  // namespace gattn
