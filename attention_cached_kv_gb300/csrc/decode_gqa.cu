// decode_gqa.cu -- one new token (l = 1) of a GQA group against a long cached
// context read through a block table: the paged decode step when 2..16 query
// heads share each KV head.
//
// [KV page, "Reusable-state"]: o_t = softmax(q_t K_{<=t}^T / sqrt(d_k)) V_{<=t},
// K_{<=t} = [K_{<t}; k_t]; [Suffix page, §5 第一步 and §6 问题四]: the context
// lives in fixed-size blocks of a pool reached through a block table.  Every
// query head of a group reads the same K/V rows, so each row is read once per
// KV head: one CTA per (sequence, KV head) of W warps, warp w taking the
// 16-key chunks w, w + W, ... of the context (W = 4; 8 for an E4M3 pool with
// one 8-head tile, where the widening doubles the work per chunk).
//
// A chunk's K and V rows (16 rows of one block and head, contiguous in the pool)
// arrive by tensor copies with 128-byte swizzle into a per-warp ring, issued by
// the warp's lane 0.  Per chunk the warp forms S^T = K q^T on
// mma.sync m16n8k16 with the keys as the 16 rows and the group's heads as the
// N (one or two 8-head tiles), q rotated in fp32 and split into bf16 hi + lo;
// keeps a running maximum and sum per head (shuffles down the key rows), moves
// P^T into the A layout by movmatrix.trans and accumulates O = P V on the same
// MMA.  At the end the W warps' (maximum, sum, O) and the new token's own key
// and value (an fp32 dot of the unrotated q and k_new: the same rotation of both
// cancels) merge in shared memory.
//
// FP8 pool ([Suffix page, §2 and the end of §5], one fp32 scale per (block,
// layer, K|V, KV head)): a ring stage holds a chunk's E4M3 rows, which the
// warp widens to f16 (exact) into one tile pair of its own and then refills
// the stage at once; q is divided by a power of two per head into the
// f16 range and split into f16 hi + lo; the K scale multiplies the fp32 logits,
// each block's V scale over the context's largest the fp32 weights, and that
// largest scale the merged output.
//
// STATS: also each cached block's attention mass per query head ([Suffix page,
// §4, §5 第三步]): per chunk and head the warp records log2 of its weight sum at
// the running maximum; they are brought to the final maximum and normaliser at
// the end and summed per block.
//
// Pages: [Suffix page] icman.com.cn news 64898;
//        [KV page] "为什么自回归推理缓存 KV，而不缓存历史 Q？".
#include <math.h>

#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace gattn {
namespace {

constexpr int kChunk = 16;           // keys per chunk
constexpr int kMaxBlocks = 512;      // cached blocks per sequence
constexpr int kMaxStatChunks = 512;  // STATS: C / 16

struct GqaParams {
  const bf16* q;
  const bf16* k_new;
  const bf16* v_new;
  bf16* out;
  const float* kv_scale;  // FP8: [num_blocks][L][2][Hkv]
  float* block_mass;      // STATS: [P][Hq][blocks_per_pair]
  PoolView pv;            // the pool (bf16, or E4M3 bytes at the same element offsets)
  const int32_t* pos_offset;
  int32_t* status;
  int Hq, Hkv, G, C;
  float scale_log2;
  double theta[64];  // RoPE frequencies (angles reduced in double)
};

// Shared memory: the warps' rings, the q tile (GN x 8 rows per panel), the
// (cos, sin) table, the block ids (and FP8 scales), the STATS log-sums and the
// mbarriers.  A bf16 ring stage holds a chunk's K tile and V tile (16 rows of
// 128 bytes per 64-column panel, 128-byte swizzle) as the tensor copies write
// them; an FP8 ring stage holds only the chunk's E4M3 rows (half a bf16
// stage), and each warp widens the chunk it computes into one K/V tile pair of
// its own.  After the chunk loop the ring
// holds the warps' partial results.  With an E4M3 pool and one 8-head tile the
// kernel runs eight warps with one or two staging stages each (the widening
// doubles the instructions per chunk, so more warps hide it); otherwise four
// warps, with three bf16 stages or four E4M3 ones.
template <int D, int GN, bool FP8, bool STATS>
struct GLayout {
  static constexpr int NP = D / 64;
  static constexpr int W = FP8 && GN == 1 ? 8 : 4;  // warps
  static constexpr int S = !FP8 ? 3 : W == 8 ? (D == 128 ? 1 : 2) : 4;  // ring stages per warp
  static constexpr uint32_t tile = kChunk * 128;
  static constexpr uint32_t k_off = 0, v_off = NP * tile;    // within a bf16 stage, or FP8 wide
  static constexpr uint32_t wide = FP8 ? 2 * NP * tile : 0;  // FP8: the warp's widened pair
  static constexpr uint32_t stage = FP8 ? 2 * kChunk * D : 2 * NP * tile;
  static constexpr uint32_t warp_bytes = wide + S * stage;
  static constexpr uint32_t ring = W * warp_bytes;
  static constexpr uint32_t q_panel = GN * 8 * 128;
  static constexpr uint32_t q_off = ring;
  static constexpr uint32_t tab_off = q_off + NP * q_panel;
  static constexpr uint32_t ids_off = tab_off + D * 4;
  static constexpr uint32_t sc_off = ids_off + kMaxBlocks * 4;
  static constexpr uint32_t lg_off = sc_off + (FP8 ? 2 * kMaxBlocks * 4 : 0);
  static constexpr uint32_t bar_off = lg_off + (STATS ? kMaxStatChunks * 16 * 4 : 0);
  static constexpr uint32_t bytes = bar_off + (W * S + 1) * 8 + 16;
  // the merge area inside the ring: per source (the W warps, the new token) and
  // head slot the maximum, the sum and O
  static constexpr uint32_t mm_off = 0, ml_off = (W + 1) * 16 * 4, mo_off = 2 * (W + 1) * 16 * 4;
  static_assert(mo_off + (W + 1) * 16 * D * 4 <= ring, "merge area");
};

template <int D, int GN, bool FP8, bool STATS>
__global__ void __launch_bounds__(GLayout<D, GN, FP8, STATS>::W * 32, FP8 ? 2 : 0)
    decode_gqa_kernel(const __grid_constant__ GqaParams prm,
                      const __grid_constant__ CUtensorMap tm_pool,
                      const __grid_constant__ CUtensorMap tm_q) {
  using L = GLayout<D, GN, FP8, STATS>;
  constexpr int NP = D / 64;
  constexpr int KS = D / 16, HK = KS / 2;
  constexpr int S = L::S;
  constexpr int kWarps = L::W, kThreads = kWarps * 32;
  constexpr float kNegInf = -INFINITY;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t base = smem_u32(smem);
  const float4* tab = reinterpret_cast<const float4*>(smem + L::tab_off);
  float2* tabw = reinterpret_cast<float2*>(smem + L::tab_off);
  int32_t* ids = reinterpret_cast<int32_t*>(smem + L::ids_off);
  float* kscale = reinterpret_cast<float*>(smem + L::sc_off);
  float* vscale = kscale + kMaxBlocks;
  float* chunk_lg = reinterpret_cast<float*>(smem + L::lg_off);  // [chunk][16 head slots]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bar_off);  // [warp][stage]
  uint64_t* qbar = full + kWarps * S;
  float* vmax_s = reinterpret_cast<float*>(qbar + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int g = blockIdx.x % prm.Hkv, p = blockIdx.x / prm.Hkv;
  const int G = prm.G, C = prm.C, bl = prm.pv.block_len, bpp = prm.pv.blocks_per_pair;
  const int nchunks = C / kChunk;

  if (tid == 0) {
    for (int i = 0; i < kWarps * S + 1; ++i) mbar_init(&full[i], 1);
    *reinterpret_cast<uint32_t*>(vmax_s) = 0u;
    fence_mbar_init();
  }
  __syncthreads();  // vmax_s starts at 0 before any thread raises it
  // head rows of the q tile past the group stay zero
  for (int idx = tid; idx < NP * (GN * 8 - G) * 8; idx += kThreads) {
    const int c = idx & 7, rest = idx >> 3, row = G + rest % (GN * 8 - G), pn = rest / (GN * 8 - G);
    sts16(base + L::q_off + pn * L::q_panel + swz128(row, c), make_uint4(0, 0, 0, 0));
  }
  bool bad = false;
  for (int b = tid; b < bpp; b += kThreads) {
    const int32_t blk = pool_block_id(prm.pv, p, b);
    const bool ok = pool_block_ok(prm.pv, blk);
    bad |= !ok;
    ids[b] = blk;
    if constexpr (FP8) {
      const int64_t si = (((int64_t)(ok ? blk : 0) * prm.pv.num_layers + prm.pv.layer) * 2) * prm.Hkv + g;
      kscale[b] = prm.kv_scale[si];
      vscale[b] = prm.kv_scale[si + prm.Hkv];
      atomicMax(reinterpret_cast<uint32_t*>(vmax_s), __float_as_uint(fmaxf(vscale[b], 0.f)));
    }
  }
  const long long pos = prm.pos_offset ? prm.pos_offset[p] : C;
  for (int j = tid; j < D / 2; j += kThreads) {
    float sn, cs;
    sincosf(rope_reduce(pos, prm.theta[j]), &sn, &cs);
    tabw[j] = make_float2(cs * prm.scale_log2, sn * prm.scale_log2);
  }
  fence_proxy_async_smem();
  bad = __syncthreads_or(bad);
  bf16* out = prm.out + ((size_t)p * prm.Hq + (size_t)g * G) * D;
  if (bad) {
    for (int e = tid; e < G * D; e += kThreads) out[e] = __float2bfloat16(0.f);
    if constexpr (STATS) {
      for (int idx = tid; idx < G * bpp; idx += kThreads)
        prm.block_mass[((size_t)p * prm.Hq + (size_t)g * G) * bpp + idx] = 0.f;
    }
    if (tid == 0) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
    return;
  }
  const float vmax = FP8 ? *vmax_s : 1.f;
  const float vinv = vmax > 0.f ? 1.f / vmax : 0.f;

  // ---- copies: the q tile (thread 0), then each warp's first chunks
  if (tid == 0) {
    mbar_arrive_expect_tx(qbar, (uint32_t)G * D * 2);
#pragma unroll
    for (int x = 0; x < NP; ++x)
      tma_load_2d(base + L::q_off + x * L::q_panel, &tm_q, qbar, 64 * x, p * prm.Hq + g * G);
  }
  const uint32_t ring_w = base + warp * L::warp_bytes;
  const uint32_t stages_w = ring_w + L::wide;  // stage s at + s * stage
  auto issue = [&](int c, int s) {  // chunk c into stage s of this warp (lane 0)
    const int key = c * kChunk, b = key / bl, t = key - b * bl;
    const int row_k =
        (int)((((int64_t)ids[b] * prm.pv.num_layers + prm.pv.layer) * 2 * prm.Hkv + g) * bl + t);
    const int row_v = row_k + prm.Hkv * bl;
    const uint32_t st = stages_w + s * L::stage;
    uint64_t* bar = &full[warp * S + s];
    if constexpr (FP8) {
      mbar_arrive_expect_tx(bar, 2u * kChunk * D);
      tma_load_2d(st, &tm_pool, bar, 0, row_k);
      tma_load_2d(st + kChunk * D, &tm_pool, bar, 0, row_v);
    } else {
      mbar_arrive_expect_tx(bar, 2u * kChunk * D * 2);
#pragma unroll
      for (int x = 0; x < NP; ++x) {
        tma_load_2d(st + L::k_off + x * L::tile, &tm_pool, bar, 64 * x, row_k);
        tma_load_2d(st + L::v_off + x * L::tile, &tm_pool, bar, 64 * x, row_v);
      }
    }
  };
  if (lane == 0)
    for (int k = 0; k < S; ++k)
      if (warp + k * kWarps < nchunks) issue(warp + k * kWarps, k);

  bool failed = !mbar_wait(qbar, 0);
  uint32_t qh[GN][KS][2], ql[GN][KS][2];
  float qf[GN];
  float snew[GN];  // warp 0: the new token's logit, head slot 8 hn + g8 (log2 units)
#pragma unroll
  for (int hn = 0; hn < GN; ++hn) {
    uint64_t rx[KS], ry[KS];
    uint32_t qr[KS][2];
    q_fragments<D, FP8>(base + L::q_off, L::q_panel, hn,
                        [&](int ks, int r) { return tab[(16 * ks + 8 * r + 2 * (lane & 3)) >> 1]; }, qh[hn],
                        ql[hn], qr, rx, ry, qf[hn]);
    snew[hn] = 0.f;
    if (warp == 0) {
      // q . k_new of the unrotated rows (the same rotation of both cancels)
      const bf16* kn = prm.k_new + ((size_t)p * prm.Hkv + g) * D;
      uint64_t dot = f2_make(0.f, 0.f);
#pragma unroll
      for (int ks = 0; ks < HK; ++ks)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int d0 = 16 * ks + 8 * r + 2 * t4;
          dot = f2_fma(rx[2 * ks + r], bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(kn + d0)), dot);
          dot = f2_fma(ry[2 * ks + r], bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(kn + d0 + D / 2)), dot);
        }
      float a, b2;
      f2_split(dot, a, b2);
      float sd = a + b2;
      sd += __shfl_xor_sync(0xffffffffu, sd, 1);
      sd += __shfl_xor_sync(0xffffffffu, sd, 2);
      snew[hn] = sd * prm.scale_log2;
    }
  }

  // ---- the chunk loop: running maximum and sum of head slots 8 hn + 2 t4 (+1)
  float m[GN][2], l[GN][2];
  float o[D / 8][4];  // rows: head slots g8 (tile 0) and 8 + g8 (tile 1)
#pragma unroll
  for (int hn = 0; hn < GN; ++hn) m[hn][0] = m[hn][1] = kNegInf, l[hn][0] = l[hn][1] = 0.f;
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
  float f0[GN], f1[GN];  // FP8: 2^e of head slots 2 t4, 2 t4 + 1
#pragma unroll
  for (int hn = 0; hn < GN; ++hn) {
    f0[hn] = FP8 ? __shfl_sync(0xffffffffu, qf[hn], 8 * t4) : 1.f;
    f1[hn] = FP8 ? __shfl_sync(0xffffffffu, qf[hn], 8 * t4 + 4) : 1.f;
  }
  int k = 0;  // chunks of this warp consumed
  for (;; ++k) {
    const int c = warp + k * kWarps;
    if (c >= nchunks || __any_sync(0xffffffffu, failed)) break;
    const int s = k % S;
    const uint32_t st = stages_w + s * L::stage;
    const uint32_t kv = FP8 ? ring_w : st;  // the chunk's K and V tiles
    if (!mbar_wait(&full[warp * S + s], (uint32_t)(k / S) & 1u)) failed = true;
    if (__any_sync(0xffffffffu, failed)) break;
    const int blk = (c * kChunk) / bl;
    if constexpr (FP8) {
      // widen the chunk's E4M3 rows to f16 in the warp's swizzled tiles (the
      // previous chunk's reads of them are done: same warp, in order)
      constexpr int CPR = D / 8, PER = 32 / CPR;
      const int cc = lane % CPR;
      for (int row = lane / CPR; row < 2 * kChunk; row += PER) {
        const uint2 raw = lds64(st + row * D + cc * 8);
        const int isv = row >= kChunk, r = row - isv * kChunk;
        sts16(kv + (isv ? L::v_off : L::k_off) + (cc >> 3) * L::tile + swz128(r, cc & 7),
              make_uint4(e4m3x2_to_f16x2(raw.x & 0xffffu), e4m3x2_to_f16x2(raw.x >> 16),
                         e4m3x2_to_f16x2(raw.y & 0xffffu), e4m3x2_to_f16x2(raw.y >> 16)));
      }
      // the staged bytes are read: refill the stage now, while this chunk is computed
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && c + S * kWarps < nchunks) issue(c + S * kWarps, s);
    }
    // S^T = K q^T: rows keys g8, g8 + 8 of the chunk; columns head slots
    float sc[GN][4];
#pragma unroll
    for (int hn = 0; hn < GN; ++hn) sc[hn][0] = sc[hn][1] = sc[hn][2] = sc[hn][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a[4];
      const int c8 = 2 * ks + (lane >> 4);
      ldsm_x4(kv + L::k_off + (c8 >> 3) * L::tile + swz128((lane & 7) + ((lane >> 3) & 1) * 8, c8 & 7), a);
#pragma unroll
      for (int hn = 0; hn < GN; ++hn) {
        mma16816<FP8>(sc[hn], a[0], a[1], a[2], a[3], qh[hn][ks][0], qh[hn][ks][1]);
        mma16816<FP8>(sc[hn], a[0], a[1], a[2], a[3], ql[hn][ks][0], ql[hn][ks][1]);
      }
    }
    const float kf = FP8 ? kscale[blk] : 1.f;
    const float vf = FP8 ? vscale[blk] * vinv : 1.f;
    uint32_t pa[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int hn = 0; hn < GN; ++hn) {
      if constexpr (FP8) {
        sc[hn][0] *= kf * f0[hn];
        sc[hn][2] *= kf * f0[hn];
        sc[hn][1] *= kf * f1[hn];
        sc[hn][3] *= kf * f1[hn];
      }
      float c0 = fmaxf(sc[hn][0], sc[hn][2]), c1 = fmaxf(sc[hn][1], sc[hn][3]);
#pragma unroll
      for (int sft = 4; sft < 32; sft <<= 1) {
        c0 = fmaxf(c0, __shfl_xor_sync(0xffffffffu, c0, sft));
        c1 = fmaxf(c1, __shfl_xor_sync(0xffffffffu, c1, sft));
      }
      const float mn0 = fmaxf(m[hn][0], c0), mn1 = fmaxf(m[hn][1], c1);
      const float al0 = ex2_approx(m[hn][0] - mn0), al1 = ex2_approx(m[hn][1] - mn1);
      const float e00 = ex2_approx(sc[hn][0] - mn0), e01 = ex2_approx(sc[hn][1] - mn1);
      const float e10 = ex2_approx(sc[hn][2] - mn0), e11 = ex2_approx(sc[hn][3] - mn1);
      float s0 = e00 + e10, s1 = e01 + e11;
#pragma unroll
      for (int sft = 4; sft < 32; sft <<= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, sft);
        s1 += __shfl_xor_sync(0xffffffffu, s1, sft);
      }
      l[hn][0] = l[hn][0] * al0 + s0;
      l[hn][1] = l[hn][1] * al1 + s1;
      m[hn][0] = mn0;
      m[hn][1] = mn1;
      if constexpr (STATS) {
        if (g8 == 0) {
          chunk_lg[c * 16 + hn * 8 + 2 * t4] = __log2f(s0) + mn0;
          chunk_lg[c * 16 + hn * 8 + 2 * t4 + 1] = __log2f(s1) + mn1;
        }
      }
      // P^T (keys x head slots) -> P (head slots x keys) in the A layout
      pa[hn] = movmatrix_trans(pack_p<FP8>(e00 * vf, e01 * vf));
      pa[hn + 2] = movmatrix_trans(pack_p<FP8>(e10 * vf, e11 * vf));
      // this lane's O rows are head slot 8 hn + g8: its factor sits in lane g8 / 2
      const float a0 = __shfl_sync(0xffffffffu, al0, g8 >> 1);
      const float a1 = __shfl_sync(0xffffffffu, al1, g8 >> 1);
      const float ar = (g8 & 1) ? a1 : a0;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        o[dn][2 * hn] *= ar;
        o[dn][2 * hn + 1] *= ar;
      }
    }
#pragma unroll
    for (int dq = 0; dq < D / 16; ++dq) {
      uint32_t bv[4];
      const int c8 = 2 * dq + (lane >> 4);
      ldsm_x4_trans(kv + L::v_off + (c8 >> 3) * L::tile + swz128((lane & 7) + ((lane >> 3) & 1) * 8, c8 & 7), bv);
      mma16816<FP8>(o[2 * dq], pa[0], pa[1], pa[2], pa[3], bv[0], bv[1]);
      mma16816<FP8>(o[2 * dq + 1], pa[0], pa[1], pa[2], pa[3], bv[2], bv[3]);
    }
    // (bf16) stage s is free: its reads come before the refill
    if constexpr (!FP8) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && c + S * kWarps < nchunks) issue(c + S * kWarps, s);
    } else {
      __syncwarp();  // every lane is done with the widened tiles before the next widening
    }
  }
  if (__any_sync(0xffffffffu, failed)) {
    if (lane == 0) {
      report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
      // wait (bounded) once for each of this warp's copies still in flight:
      // chunks k .. k + S - 1 were issued and not consumed
      for (int j = k; j < k + S && warp + j * kWarps < nchunks; ++j)
        mbar_wait(&full[warp * S + j % S], (uint32_t)(j / S) & 1u);
    }
  }

  // ---- merge: every warp's (maximum, sum, O) and the new token into the ring
  __syncthreads();
  float* mm = reinterpret_cast<float*>(smem + L::mm_off);  // [5][16]
  float* ml = reinterpret_cast<float*>(smem + L::ml_off);  // [5][16]
  float* mo = reinterpret_cast<float*>(smem + L::mo_off);  // [5][16][D]
#pragma unroll
  for (int hn = 0; hn < GN; ++hn) {
    if (g8 == 0) {
      mm[warp * 16 + hn * 8 + 2 * t4] = m[hn][0];
      mm[warp * 16 + hn * 8 + 2 * t4 + 1] = m[hn][1];
      ml[warp * 16 + hn * 8 + 2 * t4] = l[hn][0];
      ml[warp * 16 + hn * 8 + 2 * t4 + 1] = l[hn][1];
    }
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      float* row = mo + ((size_t)warp * 16 + hn * 8 + g8) * D + dn * 8 + 2 * t4;
      row[0] = o[dn][2 * hn] * vmax;
      row[1] = o[dn][2 * hn + 1] * vmax;
    }
  }
  if (warp == 0 && t4 == 0) {
    // the new token: its logit, weight 1 at its own maximum
#pragma unroll
    for (int hn = 0; hn < GN; ++hn) {
      mm[kWarps * 16 + hn * 8 + g8] = snew[hn];
      ml[kWarps * 16 + hn * 8 + g8] = 1.f;
    }
  }
  {
    const bf16* vn = prm.v_new + ((size_t)p * prm.Hkv + g) * D;
    for (int idx = tid; idx < GN * 8 * D; idx += kThreads)
      mo[(size_t)kWarps * 16 * D + idx] = __bfloat162float(vn[idx % D]);
  }
  __syncthreads();
  // out[h][col] = sum_w 2^(m_w - M) O_w / sum_w 2^(m_w - M) l_w (head h = slot h)
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int h = idx / D, col = idx - h * D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w <= kWarps; ++w) M = fmaxf(M, mm[w * 16 + h]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w <= kWarps; ++w) {
      const float f = ex2_approx(mm[w * 16 + h] - M);
      num += f * mo[((size_t)w * 16 + h) * D + col];
      den += f * ml[w * 16 + h];
    }
    out[idx] = __float2bfloat16(num / den);
  }
  if constexpr (STATS) {
    // block b's mass of head h: its chunks' log-sums at the final maximum, over the normaliser
    const int cpb = bl / kChunk;
    for (int idx = tid; idx < G * bpp; idx += kThreads) {
      const int h = idx / bpp, b = idx - h * bpp;
      float M = kNegInf;
#pragma unroll
      for (int w = 0; w <= kWarps; ++w) M = fmaxf(M, mm[w * 16 + h]);
      float den = 0.f;
#pragma unroll
      for (int w = 0; w <= kWarps; ++w) den += ex2_approx(mm[w * 16 + h] - M) * ml[w * 16 + h];
      float acc = 0.f;
      for (int c = b * cpb; c < (b + 1) * cpb; ++c) acc += ex2_approx(chunk_lg[c * 16 + h] - M);
      prm.block_mass[((size_t)p * prm.Hq + (size_t)g * G + h) * bpp + b] = acc / den;
    }
  }
}

template <int D, int GN, bool FP8, bool STATS>
int launch_d(const Problem& pb, const float* kv_scale, float* block_mass, cudaStream_t stream) {
  using L = GLayout<D, GN, FP8, STATS>;
  GqaParams prm{};
  prm.q = static_cast<const bf16*>(pb.q);
  prm.k_new = static_cast<const bf16*>(pb.k_new);
  prm.v_new = static_cast<const bf16*>(pb.v_new);
  prm.out = static_cast<bf16*>(pb.out);
  prm.kv_scale = kv_scale;
  prm.block_mass = block_mass;
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
  alignas(64) CUtensorMap tm_pool{}, tm_q{};
  const int64_t pool_rows = (int64_t)pb.num_blocks * pb.L * 2 * pb.Hkv * pb.block_len;
  int rc = FP8 ? encode_2d(&tm_pool, pb.kv_pool, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pool_rows, D, D,
                           kChunk, false)
               : encode_2d(&tm_pool, pb.kv_pool, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool_rows, D,
                           64, kChunk, true);
  if (rc == GIST_ATTN_OK)
    rc = encode_2d(&tm_q, pb.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (int64_t)pb.P * pb.Hq, D, 64,
                   pb.G, true);
  if (rc != GIST_ATTN_OK) return rc;
  const uint32_t bytes = L::bytes + 1024;  // + alignment slack
  auto kern = decode_gqa_kernel<D, GN, FP8, STATS>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  const int64_t grid = (int64_t)pb.P * pb.Hkv;
  kern<<<(unsigned)grid, L::W * 32, bytes, stream>>>(prm, tm_pool, tm_q);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

template <bool FP8, bool STATS>
int launch_shape(const Problem& pb, const float* kv_scale, float* block_mass, cudaStream_t stream) {
  const bool g2 = pb.G > 8;
  if (pb.d == 64)
    return g2 ? launch_d<64, 2, FP8, STATS>(pb, kv_scale, block_mass, stream)
              : launch_d<64, 1, FP8, STATS>(pb, kv_scale, block_mass, stream);
  if (pb.d == 128)
    return g2 ? launch_d<128, 2, FP8, STATS>(pb, kv_scale, block_mass, stream)
              : launch_d<128, 1, FP8, STATS>(pb, kv_scale, block_mass, stream);
  return GIST_ATTN_ERR_UNSUPPORTED;
}

}  // namespace

// l = 1, groups of 2..16 query heads, a cache of whole 16-row chunks in blocks
// of a multiple of 16 rows (at most 512 blocks), above the short decode's 32 keys.
bool decode_gqa_fits(const Problem& pb) {
  const int64_t pool_rows = (int64_t)pb.num_blocks * pb.L * 2 * pb.Hkv * pb.block_len;
  return pb.l == 1 && pb.G >= 2 && pb.G <= 16 && pb.C > 32 && pb.block_len % kChunk == 0 &&
         pb.blocks_per_pair <= kMaxBlocks && (pb.d == 64 || pb.d == 128) && pool_rows < 0x7fffffff &&
         (int64_t)pb.P * pb.Hq < 0x7fffffff && (int64_t)pb.P * pb.Hkv <= 0x7fffffff;
}

bool decode_gqa_stats_fits(const Problem& pb) {
  return decode_gqa_fits(pb) && pb.C / kChunk <= kMaxStatChunks;
}

int launch_decode_gqa(const Problem& pb, cudaStream_t stream) {
  return launch_shape<false, false>(pb, nullptr, nullptr, stream);
}

int launch_decode_gqa_fp8(const Problem& pb, const float* kv_scale, cudaStream_t stream) {
  return launch_shape<true, false>(pb, kv_scale, nullptr, stream);
}

int launch_decode_gqa_stats(const Problem& pb, float* block_mass, cudaStream_t stream) {
  return launch_shape<false, true>(pb, nullptr, block_mass, stream);
}

}  // namespace gattn
