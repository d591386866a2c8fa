// decode.cu -- one new token (l = 1) against a pair's cached segment.
//
// [KV page, "Reusable-state"]: o_t = softmax(q_t K_{<=t}^T / sqrt(d_k)) V_{<=t}
// with K_{<=t} = [K_{<t}; k_t]; the new token sees every cached key and its
// own.  Covers the query-gisted form of [Gist page, "能不能再进一步"] (the EOS
// token against an item-gist block and a query-gist block, both read-only, its
// own K/V never stored) and a paged cache read through a block table
// ([Suffix page, §5 第一步 and §6 问题四]).
//
// One CTA per (pair, KV head); its Hq/Hkv query heads share every key row read.
// The keys are cut into chunks of 32; warp w takes chunks w, w+4, ...; lane i of
// a chunk owns key 32c+i for the logits (one 16-byte load per 8 elements of
// its row), then the warp walks the chunk's value rows with each lane owning
// d/32 columns (coalesced rows).  Each warp keeps a running max / sum per head;
// the four warps' partial results are merged in shared memory.
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上";
//        [Suffix page] icman.com.cn news 64898;
//        [KV page] "为什么自回归推理缓存 KV，而不缓存历史 Q？".
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace gattn {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kGMax = 16;  // query heads per KV head handled by this kernel
constexpr int kMaxSmem = 227 * 1024;

struct DecodeParams {
  const bf16* q;
  const bf16* k_new;
  const bf16* v_new;
  bf16* out;
  PoolView pv;
  const int32_t* pos_offset;
  int32_t* status;
  int Hq, Hkv, G, C;
  float scale_log2;
  double theta[64];  // RoPE frequencies (angles reduced in double)
};

// shared memory: ids[bpp] | q_s[G][D] | kn_s[D] | vn_s[D] | red_m[W][G] | red_l[W][G] | red_o[W][G][D]
size_t smem_bytes(const Problem& pb) {
  size_t b = ((size_t)pb.blocks_per_pair * 4 + 15) / 16 * 16;
  b += (size_t)pb.G * pb.d * 4 + 2 * (size_t)pb.d * 4;
  b += 2 * (size_t)kWarps * pb.G * 4;
  b += (size_t)kWarps * pb.G * pb.d * 4;
  return b;
}

template <int D>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ DecodeParams prm) {
  constexpr int HALF = D / 2;
  constexpr int CPR = D / 8;   // 16-byte chunks per row
  constexpr int DPL = D / 32;  // value columns per lane
  constexpr float kNegInf = -INFINITY;

  extern __shared__ __align__(16) uint8_t smem[];
  const int G = prm.G, C = prm.C;
  int32_t* ids = reinterpret_cast<int32_t*>(smem);
  float* q_s = reinterpret_cast<float*>(smem + (prm.pv.blocks_per_pair * 4 + 15) / 16 * 16);
  float* kn_s = q_s + G * D;
  float* vn_s = kn_s + D;
  float* red_m = vn_s + D;
  float* red_l = red_m + kWarps * G;
  float* red_o = red_l + kWarps * G;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x % prm.Hkv;
  const int p = blockIdx.x / prm.Hkv;
  const int nk = C + 1;

  bool bad = false;
  for (int b = tid; b < prm.pv.blocks_per_pair; b += kThreads) {
    const int32_t blk = pool_block_id(prm.pv, p, b);
    bad |= !pool_block_ok(prm.pv, blk);
    ids[b] = blk;
  }
  // rotated, pre-scaled queries of the group; rotated new key; new value
  const long long pos = prm.pos_offset ? prm.pos_offset[p] : C;
  for (int idx = tid; idx < (G + 1) * HALF; idx += kThreads) {
    const int h = idx / HALF, j = idx - h * HALF;  // h == G: the new key
    const bf16* src = h < G ? prm.q + ((int64_t)p * prm.Hq + g * G + h) * D
                            : prm.k_new + ((int64_t)p * prm.Hkv + g) * D;
    const float x = __bfloat162float(src[j]), y = __bfloat162float(src[j + HALF]);
    float s, c;
    sincosf(rope_reduce(pos, prm.theta[j]), &s, &c);
    const float sc = h < G ? prm.scale_log2 : 1.f;
    float* dst = h < G ? q_s + h * D : kn_s;
    dst[j] = (x * c - y * s) * sc;
    dst[j + HALF] = (y * c + x * s) * sc;
  }
  for (int e = tid; e < D; e += kThreads)
    vn_s[e] = __bfloat162float(prm.v_new[((int64_t)p * prm.Hkv + g) * D + e]);
  bad = __syncthreads_or(bad);

  bf16* out = prm.out + ((int64_t)p * prm.Hq + g * G) * D;
  if (bad) {
    for (int idx = tid; idx < G * D; idx += kThreads) out[idx] = __float2bfloat16(0.f);
    if (tid == 0) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
    return;
  }

  const int bl = prm.pv.block_len;
  float m[kGMax], lsum[kGMax], o[kGMax][DPL];
#pragma unroll
  for (int h = 0; h < kGMax; ++h) {
    m[h] = kNegInf;
    lsum[h] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[h][e] = 0.f;
  }

  const int n_chunks = (nk + 31) / 32;
  for (int ch = warp; ch < n_chunks; ch += kWarps) {
    const int kappa = ch * 32 + lane;
    // ---- logits of this lane's key for every head of the group
    float s[kGMax];
#pragma unroll
    for (int h = 0; h < kGMax; ++h) s[h] = 0.f;
    if (kappa < C) {
      const int b = kappa / bl;
      const bf16* row = pool_row(prm.pv, ids[b], g, 0, kappa - b * bl);
      uint4 kr[CPR];
#pragma unroll
      for (int c = 0; c < CPR; ++c) kr[c] = ldg16(row + c * 8);
#pragma unroll
      for (int c = 0; c < CPR; ++c) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&kr[c]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 kf = bf16x2_to_float2(w[e]);
          const int col = c * 8 + 2 * e;
#pragma unroll
          for (int h = 0; h < kGMax; ++h)
            if (h < G) s[h] += q_s[h * D + col] * kf.x + q_s[h * D + col + 1] * kf.y;
        }
      }
    } else if (kappa == C) {
      for (int col = 0; col < D; ++col) {
        const float kf = kn_s[col];
#pragma unroll
        for (int h = 0; h < kGMax; ++h)
          if (h < G) s[h] += q_s[h * D + col] * kf;
      }
    }
    // ---- online softmax over the chunk, per head
    float pr[kGMax];
#pragma unroll
    for (int h = 0; h < kGMax; ++h) {
      if (h < G) {
        const float sv = kappa < nk ? s[h] : kNegInf;
        float cm = sv;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
        const float mn = fmaxf(m[h], cm);
        const float al = exp2f(m[h] - mn);
        m[h] = mn;
        pr[h] = exp2f(sv - mn);
        lsum[h] = lsum[h] * al + pr[h];
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[h][e] *= al;
      } else {
        pr[h] = 0.f;
      }
    }
    // ---- O += P V over the chunk's rows (lane owns columns lane*DPL ..)
    const int rows_here = min(32, nk - ch * 32);
    for (int kk = 0; kk < rows_here; ++kk) {
      const int key = ch * 32 + kk;
      float v[DPL];
      if (key < C) {
        const int b = key / bl;
        const bf16* row = pool_row(prm.pv, ids[b], g, 1, key - b * bl) + lane * DPL;
        if constexpr (DPL == 4) {
          const uint2 raw = *reinterpret_cast<const uint2*>(row);
          const float2 a = bf16x2_to_float2(raw.x), c2 = bf16x2_to_float2(raw.y);
          v[0] = a.x; v[1] = a.y; v[2] = c2.x; v[3] = c2.y;
        } else {
          const float2 a = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(row));
          v[0] = a.x; v[1] = a.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < DPL; ++e) v[e] = vn_s[lane * DPL + e];
      }
#pragma unroll
      for (int h = 0; h < kGMax; ++h) {
        if (h < G) {
          const float ph = __shfl_sync(0xffffffffu, pr[h], kk);
#pragma unroll
          for (int e = 0; e < DPL; ++e) o[h][e] += ph * v[e];
        }
      }
    }
  }

  // ---- merge the warps' partial results
#pragma unroll
  for (int h = 0; h < kGMax; ++h) {
    if (h < G) {
      float ls = lsum[h];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
      if (lane == 0) {
        red_m[warp * G + h] = m[h];
        red_l[warp * G + h] = ls;
      }
#pragma unroll
      for (int e = 0; e < DPL; ++e) red_o[(warp * G + h) * D + lane * DPL + e] = o[h][e];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int h = idx / D, e = idx - h * D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * G + h]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = exp2f(red_m[w * G + h] - M);  // 0 for a warp that saw no key
      num += red_o[(w * G + h) * D + e] * f;
      den += red_l[w * G + h] * f;
    }
    out[idx] = __float2bfloat16(num / den);
  }
}

template <int D>
int launch_d(const Problem& pb, cudaStream_t stream) {
  const size_t bytes = smem_bytes(pb);
  if (bytes > (size_t)kMaxSmem || pb.G > kGMax) return GIST_ATTN_ERR_UNSUPPORTED;
  DecodeParams prm{};
  prm.q = static_cast<const bf16*>(pb.q);
  prm.k_new = static_cast<const bf16*>(pb.k_new);
  prm.v_new = static_cast<const bf16*>(pb.v_new);
  prm.out = static_cast<bf16*>(pb.out);
  prm.pv = PoolView{static_cast<const bf16*>(pb.kv_pool), pb.item_ids, pb.block_table,
                    pb.blocks_per_pair, pb.block_len, pb.num_blocks, pb.L, pb.layer, pb.Hkv, pb.d};
  prm.pos_offset = pb.pos_offset;
  prm.status = pb.status;
  prm.Hq = pb.Hq;
  prm.Hkv = pb.Hkv;
  prm.G = pb.G;
  prm.C = pb.C;
  prm.scale_log2 = pb.scale_log2;
  for (int j = 0; j < 64; ++j) prm.theta[j] = pb.inv_freq_d[j];
  if (bytes > 48 * 1024 &&
      cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  const int64_t grid = (int64_t)pb.P * pb.Hkv;
  if (grid > 0x7fffffff) return GIST_ATTN_ERR_UNSUPPORTED;
  decode_kernel<D><<<(unsigned)grid, kThreads, bytes, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

}  // namespace

bool decode_fits(const Problem& pb) {
  return pb.G <= kGMax && smem_bytes(pb) <= (size_t)kMaxSmem;
}

int launch_decode(const Problem& pb, cudaStream_t stream) {
  if (pb.d == 64) return launch_d<64>(pb, stream);
  if (pb.d == 128) return launch_d<128>(pb, stream);
  return GIST_ATTN_ERR_UNSUPPORTED;
}

}  // namespace gattn
