// stage.cu -- the staged path for long new blocks behind a cached segment
// (more than 128 keys, d = 64): a pre-pass writes each pair's whole key sequence
// [cached; new] and the rotation angles of q into a caller-provided workspace,
// then the long-sequence tensor-core kernel runs on it, rotating q as it loads.
//
// [Gist page, "在线的一次 attention"]: K = cat(cache[item].K[layer], K_new),
// V likewise, the new tokens numbered after the cached positions, causal inside
// the new block.  The pre-pass writes exactly that concatenation, per pair:
//   kw [P][C + l][Hkv][64]   f16, the cached keys as stored (already rotated by
//                            their producer), then the new keys rotated
//   vw [P][C + l][Hkv][64]   bf16, the cached values, then v_new
// so that every key block of the attention is one TMA box and each key is
// rotated once per call, not once per row tile that reads it; and the angles
// of q: (cos, sin)(pos_offset[p] theta_j) per pair and (cos, sin)(i theta_j)
// per new-token index, which the attention kernel adds.  Rotated q and keys are
// rounded once to f16 (cached bf16 keys convert exactly), as in the
// single-pass tensor-core kernel.  A pair with a block id outside the pool gets
// zero values, so its output rows come out exactly 0, and the status word says
// so.
//
// One CTA per pair.  Angles: base angles (position x frequency) reduced modulo
// 2 pi in double (rope_reduce), so every int32 position keeps its accuracy;
// those of the new keys for up to 128 tokens at a time in shared memory, the
// chunk's base plus t theta_j in fp32, (cos_j, cos_j+1, sin_j, sin_j+1) per
// frequency pair.  A key chunk with a value past the f16 range is written as
// NaN, so the rows that read it come out with a non-finite softmax sum and the
// attention kernel recomputes them in fp32 from the inputs.
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上".
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace gattn {
namespace {

constexpr int kThreads = 256;
constexpr int kTabRows = 128;     // tokens per angle table
constexpr int kMaxStageBlocks = 64;  // cached blocks per pair
constexpr int kD = 64;

struct StageParams {
  const bf16* k_new;
  const bf16* v_new;
  PoolView pv;
  const int32_t* pos_offset;
  int32_t* status;
  float2* base;  // [P][32]: (cos, sin) of pos_offset[p] theta_j
  float2* rel;   // [l][32]: (cos, sin) of i theta_j
  uint16_t* kw;  // f16 bits
  bf16* vw;
  int l, Hkv, C;
  float inv_freq[32];
  double theta[32];  // the same frequencies in double
};

__device__ __forceinline__ uint32_t to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 bf16x2_f2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
// An f16 chunk, or all NaN if one element is not finite (past the f16 range).
__device__ __forceinline__ uint4 f16_chunk_or_nan(uint4 h) {
  const bool bad = (h.x & 0x7c00u) == 0x7c00u || (h.x & 0x7c000000u) == 0x7c000000u ||
                   (h.y & 0x7c00u) == 0x7c00u || (h.y & 0x7c000000u) == 0x7c000000u ||
                   (h.z & 0x7c00u) == 0x7c00u || (h.z & 0x7c000000u) == 0x7c000000u ||
                   (h.w & 0x7c00u) == 0x7c00u || (h.w & 0x7c000000u) == 0x7c000000u;
  const uint32_t nan2 = 0x7e007e00u;
  return bad ? make_uint4(nan2, nan2, nan2, nan2) : h;
}

// Rotates the 8-element chunk pair (x: elements 8 c.., y: elements 32 + 8 c..)
// of one 64-element row by the angles of table row `tr`, rounds to f16, stores
// both chunks at dst (f16 row).
__device__ __forceinline__ void rotate_store(const bf16* src, uint16_t* dst, const float4* tr, int c) {
  const uint4 x = ldg16(src + 8 * c), y = ldg16(src + 32 + 8 * c);
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
  uint32_t ox[4], oy[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float4 cs = tr[4 * c + e];  // frequencies 8 c + 2 e, 8 c + 2 e + 1
    const float2 a = bf16x2_f2(xw[e]), b = bf16x2_f2(yw[e]);
    ox[e] = to_f16x2(a.x * cs.x - b.x * cs.z, a.y * cs.y - b.y * cs.w);
    oy[e] = to_f16x2(b.x * cs.x + a.x * cs.z, b.y * cs.y + a.y * cs.w);
  }
  stg16(dst + 8 * c, f16_chunk_or_nan(make_uint4(ox[0], ox[1], ox[2], ox[3])));
  stg16(dst + 32 + 8 * c, f16_chunk_or_nan(make_uint4(oy[0], oy[1], oy[2], oy[3])));
}

__global__ void __launch_bounds__(kThreads) stage_kernel(const __grid_constant__ StageParams prm) {
  __shared__ float4 tab[kTabRows * 16];
  __shared__ float base_ang[32];
  __shared__ int32_t ids[kMaxStageBlocks];
  const int tid = threadIdx.x, p = blockIdx.x;
  const int l = prm.l, Hkv = prm.Hkv, C = prm.C, rows = C + l;
  const int bpp = prm.pv.blocks_per_pair;

  bool bad = false;
  for (int b = tid; b < bpp; b += kThreads) {
    const int32_t blk = pool_block_id(prm.pv, p, b);
    bad |= !pool_block_ok(prm.pv, blk);
    ids[b] = blk;
  }
  bad = __syncthreads_or(bad);
  if (bad && tid == 0) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
  const uint4 zero = make_uint4(0, 0, 0, 0);

  // cached rows: keys bf16 -> f16 (exact), values copied
  for (int idx = tid; idx < C * Hkv * 8; idx += kThreads) {
    const int c = idx & 7, g = (idx >> 3) % Hkv, t = (idx >> 3) / Hkv;
    const size_t o = (((size_t)p * rows + t) * Hkv + g) * kD + 8 * c;
    if (bad) {
      stg16(prm.kw + o, zero);
      stg16(prm.vw + o, zero);
      continue;
    }
    const int b = t / prm.pv.block_len, r = t - b * prm.pv.block_len;
    const uint4 k = ldg16(pool_row(prm.pv, ids[b], g, 0, r) + 8 * c);
    const uint4 v = ldg16(pool_row(prm.pv, ids[b], g, 1, r) + 8 * c);
    const uint32_t kk[4] = {k.x, k.y, k.z, k.w};
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = bf16x2_f2(kk[e]);
      h[e] = to_f16x2(f.x, f.y);
    }
    stg16(prm.kw + o, f16_chunk_or_nan(make_uint4(h[0], h[1], h[2], h[3])));
    stg16(prm.vw + o, v);
  }

  // the angles of q: this pair's base, and the rows i = p, p + P, ... of the
  // per-index table
  const int pos0 = prm.pos_offset ? prm.pos_offset[p] : C;
  if (tid < 32) {
    float s, c;
    sincosf(rope_reduce(pos0, prm.theta[tid]), &s, &c);
    prm.base[(size_t)p * 32 + tid] = make_float2(c, s);
  }
  if (tid < 32) {
    for (int t = (int)blockIdx.x; t < l; t += (int)gridDim.x) {
      float s, c;
      sincosf(rope_reduce(t, prm.theta[tid]), &s, &c);
      prm.rel[(size_t)t * 32 + tid] = make_float2(c, s);
    }
  }

  // new keys, kTabRows at a time
  for (int t0 = 0; t0 < l; t0 += kTabRows) {
    const int nt = min(kTabRows, l - t0);
    __syncthreads();  // the previous table is no longer read
    if (tid < 32) base_ang[tid] = rope_reduce((long long)pos0 + t0, prm.theta[tid]);
    __syncthreads();
    for (int idx = tid; idx < nt * 16; idx += kThreads) {
      const int t = idx >> 4, jp = idx & 15;
      float s0, c0, s1, c1;
      sincosf(fmaf((float)t, prm.inv_freq[2 * jp], base_ang[2 * jp]), &s0, &c0);
      sincosf(fmaf((float)t, prm.inv_freq[2 * jp + 1], base_ang[2 * jp + 1]), &s1, &c1);
      tab[idx] = make_float4(c0, c1, s0, s1);
    }
    __syncthreads();
    for (int idx = tid; idx < nt * Hkv * 4; idx += kThreads) {
      const int c = idx & 3, g = (idx >> 2) % Hkv, t = (idx >> 2) / Hkv;
      const size_t src = ((size_t)p * l + t0 + t) * Hkv + g;
      const size_t dst = ((size_t)p * rows + C + t0 + t) * Hkv + g;
      if (bad) {
        stg16(prm.kw + dst * kD + 8 * c, zero);
        stg16(prm.kw + dst * kD + 32 + 8 * c, zero);
        stg16(prm.vw + dst * kD + 8 * c, zero);
        stg16(prm.vw + dst * kD + 32 + 8 * c, zero);
      } else {
        rotate_store(prm.k_new + src * kD, prm.kw + dst * kD, tab + t * 16, c);
        stg16(prm.vw + dst * kD + 8 * c, ldg16(prm.v_new + src * kD + 8 * c));
        stg16(prm.vw + dst * kD + 32 + 8 * c, ldg16(prm.v_new + src * kD + 32 + 8 * c));
      }
    }
  }
}

}  // namespace

StageLayout stage_layout(const Problem& pb) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  StageLayout L{};
  const size_t rows = (size_t)pb.C + pb.l;
  const size_t kv_bytes = (size_t)pb.P * rows * pb.Hkv * 64 * 2;
  L.base_off = 0;
  L.rel_off = up((size_t)pb.P * 32 * 8);
  L.k_off = L.rel_off + up((size_t)pb.l * 32 * 8);
  L.v_off = L.k_off + up(kv_bytes);
  L.bytes = L.v_off + up(kv_bytes);
  return L;
}

bool staged_fits(const Problem& pb) {
  if (pb.d != 64 || pb.l < 2 || pb.C + pb.l <= 128 || pb.G > 128) return false;
  if (pb.blocks_per_pair > kMaxStageBlocks || pb.gist_start) return false;
  return prefill_long_grid_ok(pb, pb.C + pb.l);
}

int launch_staged(const Problem& pb, void* workspace, cudaStream_t stream) {
  const StageLayout L = stage_layout(pb);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  StageParams prm{};
  prm.k_new = static_cast<const bf16*>(pb.k_new);
  prm.v_new = static_cast<const bf16*>(pb.v_new);
  prm.pv = PoolView{static_cast<const bf16*>(pb.kv_pool), pb.item_ids, pb.block_table,
                    pb.blocks_per_pair, pb.block_len, pb.num_blocks, pb.L, pb.layer, pb.Hkv, 64};
  prm.pos_offset = pb.pos_offset;
  prm.status = pb.status;
  prm.base = reinterpret_cast<float2*>(ws + L.base_off);
  prm.rel = reinterpret_cast<float2*>(ws + L.rel_off);
  prm.kw = reinterpret_cast<uint16_t*>(ws + L.k_off);
  prm.vw = reinterpret_cast<bf16*>(ws + L.v_off);
  prm.l = pb.l;
  prm.Hkv = pb.Hkv;
  prm.C = pb.C;
  for (int j = 0; j < 32; ++j) {
    prm.inv_freq[j] = pb.inv_freq[j];
    prm.theta[j] = pb.inv_freq_d[j];
  }
  stage_kernel<<<pb.P, kThreads, 0, stream>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return GIST_ATTN_ERR_LAUNCH;
  return launch_prefill_long_on(pb, pb.q, ws + L.k_off, ws + L.v_off, pb.C, true,
                                reinterpret_cast<const float2*>(ws + L.base_off),
                                reinterpret_cast<const float2*>(ws + L.rel_off), stream);
}

}  // namespace gattn
