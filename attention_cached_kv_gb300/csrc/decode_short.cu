// decode_short.cu -- one new token (l = 1) against a short cached segment:
// the query-gisted relevance step.
//
// [Gist page, "能不能再进一步"]: with the query compressed too, only the EOS
// token is new; it attends to the k item-gist and k' query-gist positions (two
// read-only blocks) and to its own key, and its K/V are never stored.
// [KV page, "Reusable-state"]: o_t = softmax(q_t K_{<=t}^T / sqrt(d_k)) V_{<=t}.
//
// One warp per (pair, KV head).  The warp copies the group's G query rows, the
// cached K/V rows (through the pool gather) and the new value row into its own
// shared-memory region with 16-byte cp.async, rotates the new key in
// registers, and runs the whole (G <= 16) x (C + 1 <= 32) x d problem as
// tensor-core tiles: the query fragments are rotated in registers and split
// into bf16 hi + lo (two MMA passes, so the rounding of rotated q stays out of
// the logits), S = q K^T and O = P V on mma.sync m16n8k16 with fp32
// accumulation, the softmax on the S fragments with quad shuffles.  Rows are
// written straight from the accumulator fragments.  (The problem is 7 x 17 x
// 64 here; the 5th-generation MMA needs at least 64 rows.)
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上";
//        [KV page] "为什么自回归推理缓存 KV，而不缓存历史 Q？".
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace gattn {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxKeys = 32;  // C + 1
constexpr int kMaxBlocks = 32;

struct ShortParams {
  const bf16* q;
  const bf16* k_new;
  const bf16* v_new;
  bf16* out;
  PoolView pv;
  const int32_t* pos_offset;
  int32_t* status;
  int Hq, Hkv, G, C;
  int64_t units;
  float scale_log2;
  float inv_freq[64];
};

template <int D>
struct WarpRegion {  // per-warp shared memory, 128-byte swizzled rows
  static constexpr uint32_t kPanelQ = 16 * 128;         // one 64-column panel of 16 q rows
  static constexpr uint32_t kPanelKV = kMaxKeys * 128;  // one panel of 32 key rows
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + (D / 64) * kPanelQ;
  static constexpr uint32_t kV = kK + (D / 64) * kPanelKV;
  static constexpr uint32_t kTab = kV + (D / 64) * kPanelKV;  // (cos, sin) per frequency
  static constexpr uint32_t kIds = kTab + (D / 2) * 8;         // the pair's block ids
  static constexpr uint32_t kBytes = kIds + kMaxBlocks * 4;
};

template <int D>
__global__ void __launch_bounds__(kThreads) decode_short_kernel(const __grid_constant__ ShortParams prm) {
  using R = WarpRegion<D>;
  constexpr int CPR = D / 8;
  constexpr int HALF = D / 2;
  constexpr float kNegInf = -INFINITY;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t unit = (int64_t)blockIdx.x * kWarps + warp;
  if (unit >= prm.units) return;
  const int g = (int)(unit % prm.Hkv);
  const int64_t p = unit / prm.Hkv;
  const int G = prm.G, C = prm.C, NK = C + 1;
  const int bl = prm.pv.block_len;
  uint8_t* reg = smem + warp * ((R::kBytes + 1023) & ~1023u);
  const uint32_t base = smem_u32(reg);
  const uint32_t sQ = base + R::kQ, sK = base + R::kK, sV = base + R::kV;
  auto addr = [](uint32_t b, uint32_t pstride, int row, int chunk) {
    return b + (chunk >> 3) * pstride + swz128(row, chunk & 7);
  };

  // block ids of this pair (lanes < blocks_per_pair), kept in the warp's region
  int32_t* ids = reinterpret_cast<int32_t*>(reg + R::kIds);
  bool bad = false;
  if (lane < prm.pv.blocks_per_pair) {
    const int32_t blk = pool_block_id(prm.pv, (int)p, lane);
    bad = !pool_block_ok(prm.pv, blk);
    ids[lane] = blk;
  }
  bad = __any_sync(0xffffffffu, bad);
  __syncwarp();  // the ids are visible to every lane
  bf16* out = prm.out + (p * prm.Hq + (int64_t)g * G) * D;
  if (bad) {
    for (int idx = lane; idx < G * D / 8; idx += 32)
      *reinterpret_cast<uint4*>(out + idx * 8) = make_uint4(0, 0, 0, 0);
    if (lane == 0) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
    return;
  }

  // ---- copies: q rows, cached K/V rows, the new V row; zero the rest
  const bf16* qsrc = prm.q + (p * prm.Hq + (int64_t)g * G) * D;
  for (int idx = lane; idx < G * CPR; idx += 32) {
    const int row = idx / CPR, c = idx - row * CPR;
    cp_async16(addr(sQ, R::kPanelQ, row, c), qsrc + row * D + c * 8);
  }
  for (int idx = lane; idx < 2 * C * CPR; idx += 32) {
    const int kv = idx >= C * CPR;
    const int rr = idx - kv * C * CPR;
    const int kappa = rr / CPR, c = rr - kappa * CPR;
    const int bi = kappa / bl;
    cp_async16(addr(kv ? sV : sK, R::kPanelKV, kappa, c),
               pool_row(prm.pv, ids[bi], g, kv, kappa - bi * bl) + c * 8);
  }
  const bf16* vsrc = prm.v_new + (p * prm.Hkv + g) * D;
  for (int c = lane; c < CPR; c += 32) cp_async16(addr(sV, R::kPanelKV, C, c), vsrc + c * 8);
  cp_async_commit();
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int idx = lane; idx < (16 - G) * CPR; idx += 32) {
    const int row = G + idx / CPR, c = idx % CPR;
    sts16(addr(sQ, R::kPanelQ, row, c), z);
  }
  for (int idx = lane; idx < 2 * (kMaxKeys - NK) * CPR; idx += 32) {
    const int kv = idx >= (kMaxKeys - NK) * CPR;
    const int rr = idx - kv * (kMaxKeys - NK) * CPR;
    const int row = NK + rr / CPR, c = rr % CPR;
    sts16(addr(kv ? sV : sK, R::kPanelKV, row, c), z);
  }
  // cos/sin of the new token's position, and its rotated key (row C)
  const float pos = (float)(prm.pos_offset ? prm.pos_offset[p] : C);
  float2* tab = reinterpret_cast<float2*>(reg + R::kTab);
  for (int j = lane; j < HALF; j += 32) {
    float s, c;
    sincosf(pos * prm.inv_freq[j], &s, &c);
    tab[j] = make_float2(c, s);
  }
  __syncwarp();
  {
    const bf16* ksrc = prm.k_new + (p * prm.Hkv + g) * D;
    for (int c = lane; c < CPR / 2; c += 32) {
      uint4 lo = ldg16(ksrc + c * 8), hi = ldg16(ksrc + HALF + c * 8);
      uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w}, hw[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 c0 = tab[c * 8 + 2 * e], c1 = tab[c * 8 + 2 * e + 1];
        const float2 x = bf16x2_to_float2(lw[e]), y = bf16x2_to_float2(hw[e]);
        lw[e] = float2_to_bf16x2(x.x * c0.x - y.x * c0.y, x.y * c1.x - y.y * c1.y);
        hw[e] = float2_to_bf16x2(y.x * c0.x + x.x * c0.y, y.y * c1.x + x.y * c1.y);
      }
      sts16(addr(sK, R::kPanelKV, C, c), make_uint4(lw[0], lw[1], lw[2], lw[3]));
      sts16(addr(sK, R::kPanelKV, C, c + CPR / 2), make_uint4(hw[0], hw[1], hw[2], hw[3]));
    }
  }
  cp_async_wait_all();
  __syncwarp();

  // ---- q fragments (rows 0..15 = heads), rotated, scaled, split into hi + lo
  uint32_t qh[D / 16][4], ql[D / 16][4];
  {
    const int row = lane & 15;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) ldsm_x4(addr(sQ, R::kPanelQ, row, ks * 2 + (lane >> 4)), qh[ks]);
    const float sc = prm.scale_log2;
#pragma unroll
    for (int ks = 0; ks < D / 32; ++ks) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = ks * 16 + 2 * (lane & 3) + ((r & 2) ? 8 : 0);
        const float2 c0 = tab[j], c1 = tab[j + 1];
        const float2 x = bf16x2_to_float2(qh[ks][r]), y = bf16x2_to_float2(qh[ks + D / 32][r]);
        const uint64_t xr = f2_make((x.x * c0.x - y.x * c0.y) * sc, (x.y * c1.x - y.y * c1.y) * sc);
        const uint64_t yr = f2_make((y.x * c0.x + x.x * c0.y) * sc, (y.y * c1.x + x.y * c1.y) * sc);
        f2_split_bf16(xr, qh[ks][r], ql[ks][r]);
        f2_split_bf16(yr, qh[ks + D / 32][r], ql[ks + D / 32][r]);
      }
    }
  }
  // ---- S = q K^T over 32 keys (4 n-tiles)
  float s[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
    const int krow = n * 8 + (lane & 7);
#pragma unroll
    for (int k2 = 0; k2 < D / 32; ++k2) {
      uint32_t b[4];
      ldsm_x4(addr(sK, R::kPanelKV, krow, k2 * 4 + (lane >> 3)), b);
      mma_16816(s[n], qh[2 * k2], b[0], b[1]);
      mma_16816(s[n], qh[2 * k2 + 1], b[2], b[3]);
      mma_16816(s[n], ql[2 * k2], b[0], b[1]);
      mma_16816(s[n], ql[2 * k2 + 1], b[2], b[3]);
    }
  }
  // ---- softmax over the NK valid keys (rows: lane/4 and lane/4 + 8)
  float ma = kNegInf, mb = kNegInf;
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    const int key = n * 8 + 2 * (lane & 3);
    s[n][0] = key < NK ? s[n][0] : kNegInf;
    s[n][1] = key + 1 < NK ? s[n][1] : kNegInf;
    s[n][2] = key < NK ? s[n][2] : kNegInf;
    s[n][3] = key + 1 < NK ? s[n][3] : kNegInf;
    ma = max3f(ma, s[n][0], s[n][1]);
    mb = max3f(mb, s[n][2], s[n][3]);
  }
  ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
  ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
  mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
  mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
  float la = 0.f, lb = 0.f;
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    s[n][0] = ex2_approx(s[n][0] - ma);
    s[n][1] = ex2_approx(s[n][1] - ma);
    s[n][2] = ex2_approx(s[n][2] - mb);
    s[n][3] = ex2_approx(s[n][3] - mb);
    la += s[n][0] + s[n][1];
    lb += s[n][2] + s[n][3];
  }
  la += __shfl_xor_sync(0xffffffffu, la, 1);
  la += __shfl_xor_sync(0xffffffffu, la, 2);
  lb += __shfl_xor_sync(0xffffffffu, lb, 1);
  lb += __shfl_xor_sync(0xffffffffu, lb, 2);
  // ---- O = P V (2 key steps of 16)
  float o[D / 8][4];
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    uint32_t pa[4];
    pa[0] = float2_to_bf16x2(s[2 * kk][0], s[2 * kk][1]);
    pa[1] = float2_to_bf16x2(s[2 * kk][2], s[2 * kk][3]);
    pa[2] = float2_to_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
    pa[3] = float2_to_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
    const int vrow = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int dq = 0; dq < D / 16; ++dq) {
      uint32_t b[4];
      ldsm_x4_trans(addr(sV, R::kPanelKV, vrow, dq * 2 + (lane >> 4)), b);
      mma_16816(o[2 * dq], pa, b[0], b[1]);
      mma_16816(o[2 * dq + 1], pa, b[2], b[3]);
    }
  }
  // ---- rows 0..G-1 straight to global (row lane/4; rows lane/4 + 8 when G > 8)
  const int ra = lane >> 2, rb = ra + 8;
  const float ia = 1.f / la, ib = 1.f / lb;
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) {
    const int col = dn * 8 + 2 * (lane & 3);
    if (ra < G)
      *reinterpret_cast<uint32_t*>(out + (int64_t)ra * D + col) = float2_to_bf16x2(o[dn][0] * ia, o[dn][1] * ia);
    if (rb < G)
      *reinterpret_cast<uint32_t*>(out + (int64_t)rb * D + col) = float2_to_bf16x2(o[dn][2] * ib, o[dn][3] * ib);
  }
}

template <int D>
int launch_d(const Problem& pb, cudaStream_t stream) {
  ShortParams prm{};
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
  prm.units = (int64_t)pb.P * pb.Hkv;
  prm.scale_log2 = pb.scale_log2;
  for (int j = 0; j < 64; ++j) prm.inv_freq[j] = pb.inv_freq[j];
  const uint32_t per_warp = (WarpRegion<D>::kBytes + 1023) & ~1023u;
  const uint32_t bytes = kWarps * per_warp;
  if (bytes > 48 * 1024 &&
      cudaFuncSetAttribute(decode_short_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  const int64_t grid = (prm.units + kWarps - 1) / kWarps;
  if (grid > 0x7fffffff) return GIST_ATTN_ERR_UNSUPPORTED;
  decode_short_kernel<D><<<(unsigned)grid, kThreads, bytes, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

}  // namespace

bool decode_short_fits(const Problem& pb) {
  return pb.l == 1 && pb.G <= 16 && pb.C + 1 <= kMaxKeys && pb.blocks_per_pair <= kMaxBlocks &&
         (pb.d == 64 || pb.d == 128);
}

int launch_decode_short(const Problem& pb, cudaStream_t stream) {
  if (pb.d == 64) return launch_d<64>(pb, stream);
  if (pb.d == 128) return launch_d<128>(pb, stream);
  return GIST_ATTN_ERR_UNSUPPORTED;
}

}  // namespace gattn
