// decode_long.cu -- one new token (l = 1) against a long cached context read
// through a block table: the paged decode step.
//
// [KV page, "Reusable-state"]: o_t = softmax(q_t K_{<=t}^T / sqrt(d_k)) V_{<=t},
// K_{<=t} = [K_{<t}; k_t]; [Suffix page, §5 第一步 and §6 问题四]: the context
// lives in fixed-size blocks of a pool, reached through a logical -> physical
// block table.  The cost is the read of every cached K/V row ([KV page,
// "Cost"]: O(t d) per step), so the kernel is built to stream.
//
// One CTA per (sequence, KV head), four warps, sized so every CTA of a
// batch-32 x 32-head step is resident at once (no split of the key range, no
// scratch memory).  A block's rows for one head are contiguous, so the cached
// keys are streamed 16 rows at a time by 1-D bulk (TMA) copies of K and of V
// into a 3-stage shared-memory ring.  In a 16-key chunk warp w takes keys
// 4w..4w+3: eight lanes per key form the dot product with the rotated,
// pre-scaled query held in registers (fp32), the warp keeps a running max and
// sum, and each lane accumulates d/32 columns of P V.  The new token's own
// key/value join at the end; the four warps merge in shared memory.
//
// The same kernel reads an FP8 (E4M3) pool ([Suffix page, §2 and the end of §5]:
// 1-byte KV elements), one fp32 scale per (block, layer, K|V, KV head): the
// chunks are half as many bytes, widened in registers only to f16 pairs
// (cvt e4m3x2 -> f16x2) and multiplied against the f16 query slice and the
// f16 value weight with fp32 accumulation (mixed-precision FMA).  The query is
// brought into the f16 range by a power of two (folded back into the logit);
// the K scale multiplies the fp32 logit, and the V scale multiplies each
// chunk's fp32 partial P V sum, so a small scale never pushes a weight into
// f16's subnormal range.
//
// With STATS it also writes, per (sequence, head, cached block), the block's
// attention mass -- the sum of the softmax weights of its rows -- the statistic
// the eviction of [Suffix page, §5 第三步] aggregates every 64 generated tokens.
// Each warp records log2 of its share of every chunk against its running max;
// the shares are brought to the final max and normaliser at the end.
//
// A wait on a chunk that runs out (after wait_ns) ends the walk for the whole
// CTA: no further copies are issued, every copy already issued is waited for
// once more (bounded), and GIST_ATTN_STATUS_TIMEOUT is reported; the outputs
// are then unspecified.  (GIST_ATTN_FLAG_TEST_WITHHOLD withholds the first
// chunk's copy and shortens wait_ns, so a test can walk this path.)
//
// Pages: [Suffix page] icman.com.cn news 64898;
//        [KV page] "为什么自回归推理缓存 KV，而不缓存历史 Q？".
#include <math.h>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace gattn {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = 4;
constexpr int kChunk = 16;  // keys per ring stage
constexpr int kStagesBf16 = 3;  // ring depth; the fp8 ring has twice the stages (same bytes)
constexpr int kMaxBlocks = 256;
constexpr int kMaxStatChunks = 512;  // cached rows / 16 when block masses are requested

struct LongParams {
  const float* kv_scale;  // FP8 pool: [num_blocks][L][2][Hkv], else unused
  float* block_mass;      // STATS: [P][Hq][blocks_per_pair]
  const bf16* q;
  const bf16* k_new;
  const bf16* v_new;
  bf16* out;
  PoolView pv;
  const int32_t* pos_offset;
  int32_t* status;
  int Hq, Hkv, C;
  int withhold;       // test hook: do not issue chunk 0's copy
  uint64_t wait_ns;   // limit of every wait on a copy
  float scale_log2;
  double theta[64];  // RoPE frequencies (angles reduced in double)
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// acc + a * b with a, b f16 (the low halves of the two registers) and fp32 acc
__device__ __forceinline__ float fma_f16f32(uint32_t a, uint32_t b, float acc) {
  asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"((unsigned short)a), "h"((unsigned short)b));
  return acc;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v16) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)v16));
  return h;
}

template <int D, bool FP8, bool STATS>
__global__ void __launch_bounds__(kThreads, STATS ? 6 : 7)
    decode_long_kernel(const __grid_constant__ LongParams prm) {
  constexpr int HALF = D / 2;
  constexpr int QE = D / 8;        // query elements per lane (8 lanes per key)
  constexpr int VE = D / 32;       // value columns per lane
  constexpr uint32_t kRow = FP8 ? D : D * 2;  // bytes per K or V row
  constexpr uint32_t kStageBytes = 2 * kChunk * kRow;  // K rows then V rows
  constexpr int kStages = FP8 ? 2 * kStagesBf16 : kStagesBf16;
  constexpr float kNegInf = -INFINITY;

  __shared__ __align__(128) uint8_t ring[kStages * kStageBytes];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ int32_t ids[kMaxBlocks];
  __shared__ float qs[D], kn[D], vn[D];
  __shared__ float red_m[kWarps], red_l[kWarps];
  __shared__ float red_o[kWarps][D];
  __shared__ float kscale[FP8 ? kMaxBlocks : 1], vscale[FP8 ? kMaxBlocks : 1];
  __shared__ float chunk_lg[STATS ? kMaxStatChunks : 1][kWarps];  // log2 of a warp's chunk share

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x % prm.Hkv, p = blockIdx.x / prm.Hkv;
  const int C = prm.C, bl = prm.pv.block_len;
  const int n_chunks = C / kChunk;

  bool bad = false;
  for (int b = tid; b < prm.pv.blocks_per_pair; b += kThreads) {
    const int32_t blk = pool_block_id(prm.pv, p, b);
    const bool okb = pool_block_ok(prm.pv, blk);
    bad |= !okb;
    ids[b] = blk;
    if constexpr (FP8) {
      const int64_t si = (((int64_t)(okb ? blk : 0) * prm.pv.num_layers + prm.pv.layer) * 2) *
                             prm.Hkv + g;
      kscale[b] = prm.kv_scale[si];
      vscale[b] = prm.kv_scale[si + prm.Hkv];
    }
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  // rotated query (pre-scaled to log2 units), rotated new key, new value
  const long long pos = prm.pos_offset ? prm.pos_offset[p] : C;
  for (int idx = tid; idx < 2 * HALF; idx += kThreads) {
    const int which = idx / HALF, j = idx - which * HALF;  // 0: q, 1: k_new
    const bf16* src = which == 0 ? prm.q + ((int64_t)p * prm.Hq + g) * D
                                 : prm.k_new + ((int64_t)p * prm.Hkv + g) * D;
    const float x = __bfloat162float(src[j]), y = __bfloat162float(src[j + HALF]);
    float s, c;
    sincosf(rope_reduce(pos, prm.theta[j]), &s, &c);
    const float sc = which == 0 ? prm.scale_log2 : 1.f;
    float* dst = which == 0 ? qs : kn;
    dst[j] = (x * c - y * s) * sc;
    dst[j + HALF] = (y * c + x * s) * sc;
  }
  for (int e = tid; e < D; e += kThreads)
    vn[e] = __bfloat162float(prm.v_new[((int64_t)p * prm.Hkv + g) * D + e]);
  bad = __syncthreads_or(bad);
  bf16* out = prm.out + ((int64_t)p * prm.Hq + g) * D;
  if (bad) {
    for (int e = tid; e < D; e += kThreads) out[e] = __float2bfloat16(0.f);
    if constexpr (STATS) {
      float* mass = prm.block_mass + ((int64_t)p * prm.Hq + g) * prm.pv.blocks_per_pair;
      for (int b = tid; b < prm.pv.blocks_per_pair; b += kThreads) mass[b] = 0.f;
    }
    if (tid == 0) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
    return;
  }

  const uint32_t ring0 = smem_u32(ring);
  auto issue = [&](int ci) {  // chunk ci -> stage ci % kStages (thread 0)
    const int s = ci % kStages;
    const int key = ci * kChunk, b = key / bl, t = key - b * bl;
    mbar_arrive_expect_tx(&full[s], kStageBytes);
    const bf16* krow = pool_row(prm.pv, ids[b], g, 0, t);
    const bf16* vrow = pool_row(prm.pv, ids[b], g, 1, t);
    if constexpr (FP8) {  // the same element offsets, one byte per element
      const uint8_t* p8 = reinterpret_cast<const uint8_t*>(prm.pv.pool);
      krow = reinterpret_cast<const bf16*>(p8 + (krow - prm.pv.pool));
      vrow = reinterpret_cast<const bf16*>(p8 + (vrow - prm.pv.pool));
    }
    bulk_g2s(ring0 + s * kStageBytes, krow, kChunk * kRow, &full[s]);
    bulk_g2s(ring0 + s * kStageBytes + kChunk * kRow, vrow, kChunk * kRow, &full[s]);
  };
  int issued = 0;  // thread 0: chunks whose copies were issued (0 .. issued - 1)
  if (tid == 0) {
    for (int ci = 0; ci < kStages && ci < n_chunks; ++ci)
      if (!(prm.withhold && ci == 0)) issue(ci);
    issued = min(kStages, n_chunks);
  }

  // this lane's slice of the query: elements (lane % 8) * QE ..
  const int kg = lane >> 3, sl = lane & 7;
  float qr[QE];
#pragma unroll
  for (int e = 0; e < QE; ++e) qr[e] = qs[sl * QE + e];
  // FP8: the query slice as f16 (low half of each register), for the mixed
  // f16 x f16 + fp32 products against keys widened only to f16
  uint32_t qh[FP8 ? QE : 1];
  float qfac = 1.f;  // FP8: the power of two the f16 query slice was divided by
  if constexpr (FP8) {
    float mx = 0.f;
#pragma unroll
    for (int e = 0; e < QE; ++e) mx = fmaxf(mx, fabsf(qr[e]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    const int ex = mx >= 16384.f ? ilogbf(mx) - 13 : 0;
    qfac = ldexpf(1.f, ex);
    const float inv = ldexpf(1.f, -ex);
#pragma unroll
    for (int e = 0; e < QE; ++e) {
      const __half hq = __float2half_rn(qr[e] * inv);
      qh[e] = *reinterpret_cast<const unsigned short*>(&hq);
    }
  }
  float m = kNegInf, lsum = 0.f, o[VE], last_share = kNegInf;
#pragma unroll
  for (int e = 0; e < VE; ++e) o[e] = 0.f;

  // bf16 pool: one key per 8-lane group: logit s (all 8 lanes), then the warp's
  // online update
  auto consume = [&](float s_key, bool valid, const uint8_t* vrows) {
    float sv = valid ? s_key : kNegInf;
    float cm = fmaxf(sv, __shfl_xor_sync(0xffffffffu, sv, 8));
    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
    const float mn = fmaxf(m, cm);
    const float al = ex2_approx(m - mn);
    const float pk = ex2_approx(sv - mn);  // this group's key weight
    m = mn;
    float ps = pk + __shfl_xor_sync(0xffffffffu, pk, 8);
    ps += __shfl_xor_sync(0xffffffffu, ps, 16);
    lsum = lsum * al + ps;
    last_share = ps > 0.f ? __log2f(ps) + mn : kNegInf;
#pragma unroll
    for (int e = 0; e < VE; ++e) o[e] *= al;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float pj = __shfl_sync(0xffffffffu, pk, j * 8);
      const uint8_t* vr = vrows + j * kRow + lane * VE * 2;
      if constexpr (VE == 4) {
        const uint2 raw = *reinterpret_cast<const uint2*>(vr);
        const float2 a = bf16x2_to_float2(raw.x), b2 = bf16x2_to_float2(raw.y);
        o[0] += pj * a.x; o[1] += pj * a.y; o[2] += pj * b2.x; o[3] += pj * b2.y;
      } else {
        const float2 a = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(vr));
        o[0] += pj * a.x; o[1] += pj * a.y;
      }
    }
  };

  bool failed = false;
  int consumed = 0;  // chunks whose stages this CTA has finished with
  if constexpr (FP8) {
    // Two 16-key chunks per step (an fp8 chunk is half the bytes of a bf16 one):
    // one online-softmax update and one barrier per 8 keys of a warp.
    auto kdot = [&](const uint8_t* stage) {
      const uint8_t* krow = stage + (warp * 4 + kg) * kRow + sl * QE;
      uint32_t w[QE / 4];
      if constexpr (QE == 16) {
        const uint4 raw = *reinterpret_cast<const uint4*>(krow);
        w[0] = raw.x; w[1] = raw.y; w[2] = raw.z; w[3] = raw.w;
      } else {
        const uint2 raw = *reinterpret_cast<const uint2*>(krow);
        w[0] = raw.x; w[1] = raw.y;
      }
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < QE / 4; ++e) {
        const uint32_t k0 = e4m3x2_to_f16x2(w[e] & 0xffffu), k1 = e4m3x2_to_f16x2(w[e] >> 16);
        acc = fma_f16f32(qh[4 * e], k0, acc);
        acc = fma_f16f32(qh[4 * e + 1], k0 >> 16, acc);
        acc = fma_f16f32(qh[4 * e + 2], k1, acc);
        acc = fma_f16f32(qh[4 * e + 3], k1 >> 16, acc);
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      return acc;
    };
    auto vacc = [&](const uint8_t* stage, float pk, float vsc) {
      const uint8_t* vrows = stage + kChunk * kRow + warp * 4 * kRow;
      float t[VE];
#pragma unroll
      for (int e = 0; e < VE; ++e) t[e] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half ph = __float2half_rn(__shfl_sync(0xffffffffu, pk, j * 8));
        const uint32_t p16 = *reinterpret_cast<const unsigned short*>(&ph);
        const uint8_t* vr = vrows + j * kRow + lane * VE;
        if constexpr (VE == 4) {
          const uint32_t raw = *reinterpret_cast<const uint32_t*>(vr);
          const uint32_t a = e4m3x2_to_f16x2(raw & 0xffffu), b2 = e4m3x2_to_f16x2(raw >> 16);
          t[0] = fma_f16f32(p16, a, t[0]);
          t[1] = fma_f16f32(p16, a >> 16, t[1]);
          t[2] = fma_f16f32(p16, b2, t[2]);
          t[3] = fma_f16f32(p16, b2 >> 16, t[3]);
        } else {
          const uint32_t a = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(vr));
          t[0] = fma_f16f32(p16, a, t[0]);
          t[1] = fma_f16f32(p16, a >> 16, t[1]);
        }
      }
#pragma unroll
      for (int e = 0; e < VE; ++e) o[e] = fmaf(vsc, t[e], o[e]);
    };
    for (int ci = 0; ci < n_chunks; ci += 2) {
      const bool two = ci + 1 < n_chunks;  // uniform
      const int s0 = ci % kStages, s1 = (ci + 1) % kStages;
      if (!mbar_wait(&full[s0], (uint32_t)(ci / kStages) & 1u, prm.wait_ns)) failed = true;
      if (two && !failed && !mbar_wait(&full[s1], (uint32_t)((ci + 1) / kStages) & 1u, prm.wait_ns))
        failed = true;
      if (__syncthreads_or(failed)) {
        failed = true;
        break;
      }
      const uint8_t* st0 = ring + s0 * kStageBytes;
      const uint8_t* st1 = ring + s1 * kStageBytes;
      const int b0 = (ci * kChunk) / bl, b1 = ((ci + 1) * kChunk) / bl;
      const float x0 = kdot(st0) * (kscale[b0] * qfac);
      const float x1 = two ? kdot(st1) * (kscale[b1] * qfac) : kNegInf;
      float cm = fmaxf(x0, x1);
      cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 8));
      cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
      const float mn = fmaxf(m, cm);
      const float al = ex2_approx(m - mn);
      const float p0 = ex2_approx(x0 - mn), p1 = ex2_approx(x1 - mn);
      m = mn;
      float ps0 = p0 + __shfl_xor_sync(0xffffffffu, p0, 8);
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, 16);
      float ps1 = p1 + __shfl_xor_sync(0xffffffffu, p1, 8);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, 16);
      lsum = lsum * al + ps0 + ps1;
#pragma unroll
      for (int e = 0; e < VE; ++e) o[e] *= al;
      vacc(st0, p0, vscale[b0]);
      if (two) vacc(st1, p1, vscale[b1]);
      if constexpr (STATS) {
        if (lane == 0) {
          chunk_lg[ci][warp] = ps0 > 0.f ? __log2f(ps0) + mn : kNegInf;
          if (two) chunk_lg[ci + 1][warp] = ps1 > 0.f ? __log2f(ps1) + mn : kNegInf;
        }
      }
      __syncthreads();  // every warp is done with both stages
      consumed = ci + (two ? 2 : 1);
      if (tid == 0) {
        if (ci + kStages < n_chunks) issue(ci + kStages);
        if (ci + 1 + kStages < n_chunks) issue(ci + 1 + kStages);
        issued = min(n_chunks, consumed + kStages);
      }
    }
  } else {
    for (int ci = 0; ci < n_chunks; ++ci) {
      const int s = ci % kStages;
      if (__syncthreads_or(!mbar_wait(&full[s], (uint32_t)(ci / kStages) & 1u, prm.wait_ns))) {
        failed = true;
        break;
      }
      const uint8_t* stage = ring + s * kStageBytes;
      float acc = 0.f;
      const uint8_t* krow = stage + (warp * 4 + kg) * kRow + sl * QE * 2;
#pragma unroll
      for (int v = 0; v < QE / 8; ++v) {
        const uint4 raw = *reinterpret_cast<const uint4*>(krow + v * 16);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 kf = bf16x2_to_float2(w[e]);
          acc = fmaf(qr[v * 8 + 2 * e], kf.x, acc);
          acc = fmaf(qr[v * 8 + 2 * e + 1], kf.y, acc);
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      consume(acc, true, stage + kChunk * kRow + warp * 4 * kRow);
      if constexpr (STATS) {
        if (lane == 0) chunk_lg[ci][warp] = last_share;
      }
      __syncthreads();  // every warp is done with stage s
      consumed = ci + 1;
      if (tid == 0) {
        if (ci + kStages < n_chunks) issue(ci + kStages);
        issued = min(n_chunks, consumed + kStages);
      }
    }
  }
  // the new token's own key and value (warp 0, group 0)
  if (warp == 0) {
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < QE; ++e) acc = fmaf(qr[e], kn[sl * QE + e], acc);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    // every lane holds the full dot product of q with the new key
    const float mn = fmaxf(m, acc);
    const float al = ex2_approx(m - mn);
    const float pnew = ex2_approx(acc - mn);
    m = mn;
    lsum = lsum * al + pnew;
#pragma unroll
    for (int e = 0; e < VE; ++e) o[e] = o[e] * al + pnew * vn[lane * VE + e];
  }
  if (lane == 0) {
    red_m[warp] = m;
    red_l[warp] = lsum;
  }
#pragma unroll
  for (int e = 0; e < VE; ++e) red_o[warp][lane * VE + e] = o[e];
  __syncthreads();
  for (int e = tid; e < D; e += kThreads) {
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = ex2_approx(red_m[w] - M);
      num += red_o[w][e] * f;
      den += red_l[w] * f;
    }
    out[e] = __float2bfloat16(num / den);
  }
  if constexpr (STATS) {
    // chunk share at the final max M, over the final normaliser L
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) L += red_l[w] * ex2_approx(red_m[w] - M);
    const float invL = 1.f / L;
    const int cpb = bl / kChunk;  // chunks per block
    float* mass = prm.block_mass + ((int64_t)p * prm.Hq + g) * prm.pv.blocks_per_pair;
    for (int b = tid; b < prm.pv.blocks_per_pair; b += kThreads) {
      float acc = 0.f;
      for (int c = b * cpb; c < (b + 1) * cpb; ++c)
#pragma unroll
        for (int w = 0; w < kWarps; ++w) acc += ex2_approx(chunk_lg[c][w] - M);
      mass[b] = acc * invL;
    }
  }
  if (failed && tid == 0) {
    report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
    // every copy issued and not consumed lands in its stage before the CTA
    // leaves (a withheld one is skipped): one more bounded wait each
    for (int ci = consumed; ci < issued; ++ci)
      if (!(prm.withhold && ci == 0)) mbar_wait(&full[ci % kStages], (uint32_t)(ci / kStages) & 1u, prm.wait_ns);
  }
}

template <int D, bool FP8, bool STATS>
int launch_d(const Problem& pb, const float* kv_scale, float* block_mass, cudaStream_t stream) {
  LongParams prm{};
  prm.kv_scale = kv_scale;
  prm.block_mass = block_mass;
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
  prm.C = pb.C;
  prm.scale_log2 = pb.scale_log2;
  for (int j = 0; j < 64; ++j) prm.theta[j] = pb.inv_freq_d[j];
  prm.withhold = (pb.flags & GIST_ATTN_FLAG_TEST_WITHHOLD) ? 1 : 0;
  prm.wait_ns = prm.withhold ? 20000000ull : kWaitLimitNs;
  const int64_t grid = (int64_t)pb.P * pb.Hkv;
  if (grid > 0x7fffffff) return GIST_ATTN_ERR_UNSUPPORTED;
  decode_long_kernel<D, FP8, STATS><<<(unsigned)grid, kThreads, 0, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

}  // namespace

// MHA decode over a long cache whose blocks hold whole 16-row chunks.
bool decode_long_fits(const Problem& pb) {
  return pb.l == 1 && pb.G == 1 && pb.C >= 64 && pb.block_len % kChunk == 0 &&
         pb.blocks_per_pair <= kMaxBlocks && (pb.d == 64 || pb.d == 128);
}

int launch_decode_long(const Problem& pb, cudaStream_t stream) {
  if (pb.d == 64) return launch_d<64, false, false>(pb, nullptr, nullptr, stream);
  if (pb.d == 128) return launch_d<128, false, false>(pb, nullptr, nullptr, stream);
  return GIST_ATTN_ERR_UNSUPPORTED;
}

int launch_decode_long_fp8(const Problem& pb, const float* kv_scale, cudaStream_t stream) {
  if (pb.d == 64) return launch_d<64, true, false>(pb, kv_scale, nullptr, stream);
  if (pb.d == 128) return launch_d<128, true, false>(pb, kv_scale, nullptr, stream);
  return GIST_ATTN_ERR_UNSUPPORTED;
}

bool decode_long_stats_fits(const Problem& pb) {
  return decode_long_fits(pb) && pb.C / kChunk <= kMaxStatChunks;
}

int launch_decode_long_stats(const Problem& pb, float* block_mass, cudaStream_t stream) {
  if (pb.d == 64) return launch_d<64, false, true>(pb, nullptr, block_mass, stream);
  if (pb.d == 128) return launch_d<128, false, true>(pb, nullptr, block_mass, stream);
  return GIST_ATTN_ERR_UNSUPPORTED;
}

}  // namespace gattn
