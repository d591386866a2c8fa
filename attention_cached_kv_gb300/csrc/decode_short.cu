// decode_short.cu -- one new token (l = 1) against a short cached segment:
// the query-gisted relevance step.
//
// [Gist page, "能不能再进一步"]: with the query compressed too, only the EOS
// token is new; it attends to the k item-gist and k' query-gist positions (two
// read-only blocks) and to its own key, and its K/V are never stored.
// [KV page, "Reusable-state"]: o_t = softmax(q_t K_{<=t}^T / sqrt(d_k)) V_{<=t}.
//
// Persistent warps, one (pair, KV head) unit at a time, two units in flight per
// warp: while a warp computes unit n from one shared-memory buffer, the 16-byte
// cp.async copies of unit n+1 (its cached K/V rows through the pool gather, its
// new key and value rows) fill the other buffer, its query rows travel straight
// into registers in the mma fragment layout, and the block ids of unit n+2 are
// on their way.  A unit is (G <= 16) x (C + 1 <= 32) x d: the query fragments
// are rotated in registers and split into bf16 hi + lo (two MMA passes, so the
// rounding of rotated q stays out of the logits), S = q K^T and O = P V run on
// mma.sync (m16n8k16, and m16n8k8 for a last 8-key step) with fp32
// accumulation, the softmax on the S fragments with quad shuffles; rows are
// written straight from the accumulator fragments.  (The problem is 7 x 17 x 64
// here; the 5th-generation MMA needs at least 64 rows.)
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
  int kvr;          // key rows per buffer: C + 1 rounded up to 8
  uint32_t region;  // bytes of one warp's shared memory
  int units;        // P * Hkv (below 2^31)
  float scale_log2;
  double theta[64];  // RoPE frequencies (angles reduced in double)
};

// One warp's shared memory: two buffers, each with the K panels then the V
// panels (kvr rows of 128 bytes, 128-byte swizzle), then the (cos, sin) table of
// the new token's position.
template <int D>
struct Region {
  static constexpr int NP = D / 64;
  __host__ __device__ static uint32_t panel(int kvr) { return (uint32_t)kvr * 128; }
  __host__ __device__ static uint32_t buf(int kvr) { return 2u * NP * panel(kvr); }
  __host__ __device__ static uint32_t tab(int kvr) { return 2 * buf(kvr); }
  __host__ __device__ static uint32_t bars(int kvr) { return tab(kvr) + (D / 2) * 8; }  // 2 mbarriers
  // rounded to 1 KiB so that every buffer of every warp starts on a swizzle atom
  __host__ __device__ static uint32_t bytes(int kvr) { return (bars(kvr) + 16 + 1023) & ~1023u; }
};

// D(16x8) += A(16x8, bf16, row) * B(8x8, bf16, col)
__device__ __forceinline__ void mma_1688(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6},"
      " {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

__device__ __forceinline__ uint32_t ldg32(const bf16* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// G8: the group has at most 8 query heads, so rows 8..15 of every 16-row
// fragment are zero and their work is left out at compile time.
// TMA: a unit's rows arrive by tensor copies issued by one lane (cached blocks of
// a multiple of 8 rows, each (block, K|V) a {64, block_len} box, the new key and
// value {64, 1} boxes), completing on the buffer's mbarrier; otherwise every lane
// issues 16-byte cp.async copies.
template <int D, bool G8, bool TMA>
__global__ void __launch_bounds__(kThreads) decode_short_kernel(const __grid_constant__ ShortParams prm,
                                                                const __grid_constant__ CUtensorMap tm_pool,
                                                                const __grid_constant__ CUtensorMap tm_kn,
                                                                const __grid_constant__ CUtensorMap tm_vn) {
  using R = Region<D>;
  constexpr int NP = D / 64;
  constexpr int CPR = D / 8;
  constexpr int HALF = D / 2;
  constexpr int KS = D / 16;  // k-steps of the q fragments
  constexpr float kNegInf = -INFINITY;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = gridDim.x * kWarps;
  int u = blockIdx.x * kWarps + warp;
  if (u >= prm.units) return;  // warp-uniform; nothing below synchronises the CTA
  const int G = prm.G, C = prm.C, NK = C + 1, kvr = prm.kvr;
  const int bpp = prm.pv.blocks_per_pair, bl = prm.pv.block_len;
  uint8_t* reg = smem + warp * prm.region;
  const uint32_t base = smem_u32(reg);
  const uint32_t pnl = R::panel(kvr), bufb = R::buf(kvr);
  float2* tab = reinterpret_cast<float2*>(reg + R::tab(kvr));
  uint64_t* kvbar = reinterpret_cast<uint64_t*>(reg + R::bars(kvr));  // one per buffer (TMA)
  if (TMA) {
    if ((base & 1023u) != 0) {  // the swizzle atoms need 1 KiB alignment: never expected
      if (lane == 0) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
      return;
    }
    if (lane == 0) {
      mbar_init(&kvbar[0], 1);
      mbar_init(&kvbar[1], 1);
      fence_mbar_init();
    }
    __syncwarp();
  }
  auto kaddr = [&](int b, int row, int c) {
    return base + b * bufb + (c >> 3) * pnl + swz128(row, c & 7);
  };
  auto vaddr = [&](int b, int row, int c) {
    return base + b * bufb + (NP + (c >> 3)) * pnl + swz128(row, c & 7);
  };

  // rows past the keys stay zero in both buffers (no copy writes them)
  if (kvr > NK) {
    const int pad = kvr - NK;
    for (int idx = lane; idx < 2 * 2 * pad * CPR; idx += 32) {
      const int c = idx % CPR, rest = idx / CPR;
      const int row = NK + rest % pad, kv = (rest / pad) & 1, b = rest / (2 * pad);
      sts16(kv ? vaddr(b, row, c) : kaddr(b, row, c), make_uint4(0, 0, 0, 0));
    }
  }
  // (cos, sin) of the new token's position: lane j keeps frequencies j (and
  // j + 32) in registers for the key; the table holds them times the softmax
  // scale for the query fragments
  float kcos[HALF / 32], ksin[HALF / 32];
  auto build_tab = [&](int pos) {
#pragma unroll
    for (int e = 0; e < HALF / 32; ++e) {
      const int j = lane + 32 * e;
      sincosf(rope_reduce(pos, prm.theta[j]), &ksin[e], &kcos[e]);
      tab[j] = make_float2(kcos[e] * prm.scale_log2, ksin[e] * prm.scale_log2);
    }
    __syncwarp();
  };
  const bool fixed_pos = prm.pos_offset == nullptr;
  if (fixed_pos) build_tab(C);

  // block id of the unit's lane-th block (lanes < blocks_per_pair)
  auto load_id = [&](int v) -> int32_t {
    return (v < prm.units && lane < bpp) ? pool_block_id(prm.pv, v / prm.Hkv, lane) : 0;
  };
  // cp.async of unit v's rows into buffer b; true (warp-uniform) if one of its
  // block ids is out of range (its cached rows are then not copied)
  auto issue = [&](int p, int g, int b, int32_t id) -> bool {
    const bool bad = __any_sync(0xffffffffu, lane < bpp && !pool_block_ok(prm.pv, id));
    if (TMA) {
      const uint32_t buf = base + b * bufb;
      if (lane == 0)
        mbar_arrive_expect_tx(&kvbar[b], (bad ? 0u : (uint32_t)bpp * 2 * bl * 128 * NP) + 2u * 128 * NP);
      for (int bi = 0; bi < bpp; ++bi) {  // uniform loop: the shuffle is safe
        const int32_t blk = __shfl_sync(0xffffffffu, id, bi);
        if (lane == 0 && !bad) {
          const int row_k = (int)((((int64_t)blk * prm.pv.num_layers + prm.pv.layer) * 2 * prm.Hkv + g) * bl);
          const int row_v = row_k + prm.Hkv * bl;
#pragma unroll
          for (int x = 0; x < NP; ++x) {
            tma_load_2d(buf + x * pnl + bi * bl * 128, &tm_pool, &kvbar[b], 64 * x, row_k);
            tma_load_2d(buf + (NP + x) * pnl + bi * bl * 128, &tm_pool, &kvbar[b], 64 * x, row_v);
          }
        }
      }
      if (lane == 0) {
#pragma unroll
        for (int x = 0; x < NP; ++x) {
          tma_load_2d(buf + x * pnl + C * 128, &tm_kn, &kvbar[b], 64 * x, p * prm.Hkv + g);
          tma_load_2d(buf + (NP + x) * pnl + C * 128, &tm_vn, &kvbar[b], 64 * x, p * prm.Hkv + g);
        }
      }
      return bad;
    }
    constexpr int kStep = 32 / CPR;  // rows per pass of the warp
    const int c = lane % CPR, r0 = lane / CPR;
    if (!bad) {
      // this lane's chunk column c of rows r0, r0 + kStep, ... of every block;
      // a block's V rows sit Hkv * block_len rows after its K rows
      const uint32_t col = base + b * bufb + (c >> 3) * pnl;
      const uint32_t v_off = NP * pnl;
      const int64_t v_gap = (int64_t)prm.Hkv * bl * D;
      for (int bi = 0; bi < bpp; ++bi) {  // uniform loop: the shuffle is safe
        const int32_t blk = __shfl_sync(0xffffffffu, id, bi);
        const bf16* src = pool_row(prm.pv, blk, g, 0, r0) + c * 8;
        for (int row = bi * bl + r0; row < (bi + 1) * bl; row += kStep, src += kStep * D) {
          const uint32_t dst = col + swz128(row, c & 7);
          cp_async16(dst, src);
          cp_async16(dst + v_off, src + v_gap);
        }
      }
    }
    // the new token's raw key (rotated later) and its value: row C
    const size_t nrow = ((size_t)p * prm.Hkv + g) * D;
    for (int c2 = lane; c2 < 2 * CPR; c2 += 32) {
      if (c2 < CPR)
        cp_async16(kaddr(b, C, c2), prm.k_new + nrow + c2 * 8);
      else
        cp_async16(vaddr(b, C, c2 - CPR), prm.v_new + nrow + (c2 - CPR) * 8);
    }
    cp_async_commit();
    return bad;
  };
  // unit v's query rows (heads) lane/4 and lane/4 + 8 of its group in the mma
  // A-fragment layout: columns ks*16 + 2(lane%4) + {0, 1} and + 8
  auto load_q = [&](int p, int g, uint32_t (&a)[KS][4]) {
    const bf16* q0 = prm.q + ((size_t)p * prm.Hq + (size_t)g * G) * D + 2 * (lane & 3);
    const int ra = lane >> 2, rb = ra + 8;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      a[ks][0] = ra < G ? ldg32(q0 + (size_t)ra * D + ks * 16) : 0u;
      a[ks][2] = ra < G ? ldg32(q0 + (size_t)ra * D + ks * 16 + 8) : 0u;
      a[ks][1] = (!G8 && rb < G) ? ldg32(q0 + (size_t)rb * D + ks * 16) : 0u;
      a[ks][3] = (!G8 && rb < G) ? ldg32(q0 + (size_t)rb * D + ks * 16 + 8) : 0u;
    }
  };

  // ---- prologue: unit u's copies and query; the next unit's block ids
  uint32_t qcur[KS][4];
  int p = u / prm.Hkv, g = u - p * prm.Hkv;
  bool bad_cur = issue(p, g, 0, load_id(u));
  load_q(p, g, qcur);
  int un = u + W;
  int pn = un / prm.Hkv, gn = un - pn * prm.Hkv;
  int32_t id_next = load_id(un);

  for (int n = 0;; ++n) {
    const int b = n & 1;
    // ---- unit un's copies into the other buffer (free since the last unit),
    // its query into registers, and the block ids of the unit after it
    uint32_t qnext[KS][4];
    bool bad_next = false;
    const bool more = un < prm.units;
    if (more) {
      bad_next = issue(pn, gn, b ^ 1, id_next);
      load_q(pn, gn, qnext);
      id_next = load_id(un + W);
      if (!TMA) cp_async_wait_group<1>();
    } else if (!TMA) {
      cp_async_wait_group<0>();
    }
    if (TMA) {  // unit u's copies are the ((n / 2) + 1)-th phase of its buffer's barrier
      if (!mbar_wait(&kvbar[b], (uint32_t)(n >> 1) & 1u) && lane == 0)
        report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
    }
    __syncwarp();  // every lane's copies of unit u have landed

    // ---- unit u = (pair p, KV head g)
    bf16* out = prm.out + ((size_t)p * prm.Hq + (size_t)g * G) * D;
    if (bad_cur) {
      for (int idx = lane; idx < G * CPR; idx += 32)
        *reinterpret_cast<uint4*>(out + idx * 8) = make_uint4(0, 0, 0, 0);
      if (lane == 0) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
    } else {
      if (!fixed_pos) build_tab(prm.pos_offset[p]);
      // the new key (row C), rotated in place: lane j takes frequencies j, j + 32
#pragma unroll
      for (int e = 0; e < HALF / 32; ++e) {
        const int j = lane + 32 * e;
        const float2 cs = make_float2(kcos[e], ksin[e]);
        const uint32_t ax = kaddr(b, C, j >> 3) + (j & 7) * 2;
        const uint32_t ay = kaddr(b, C, (j + HALF) >> 3) + (j & 7) * 2;
        uint16_t xb, yb;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(xb) : "r"(ax));
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(yb) : "r"(ay));
        const float x = __uint_as_float((uint32_t)xb << 16), y = __uint_as_float((uint32_t)yb << 16);
        const bf16 xr = __float2bfloat16_rn(x * cs.x - y * cs.y);
        const bf16 yr = __float2bfloat16_rn(y * cs.x + x * cs.y);
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(ax), "h"(*reinterpret_cast<const uint16_t*>(&xr)));
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(ay), "h"(*reinterpret_cast<const uint16_t*>(&yr)));
      }
      __syncwarp();

      // ---- q fragments: rotated, scaled, split into hi + lo
      uint32_t qh[KS][4], ql[KS][4];
#pragma unroll
      for (int ks = 0; ks < KS / 2; ++ks) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (G8 && (r & 1)) {  // rows 8..15
            qh[ks][r] = ql[ks][r] = qh[ks + KS / 2][r] = ql[ks + KS / 2][r] = 0u;
            continue;
          }
          const int j = ks * 16 + 2 * (lane & 3) + ((r & 2) ? 8 : 0);
          const float4 cs = *reinterpret_cast<const float4*>(&tab[j]);  // (c_j, s_j, c_j+1, s_j+1)
          const uint64_t c = f2_make(cs.x, cs.z), sn = f2_make(cs.y, cs.w);
          const uint64_t x = bf16x2_to_f2(qcur[ks][r]), y = bf16x2_to_f2(qcur[ks + KS / 2][r]);
          f2_split_bf16(f2_sub(f2_mul(x, c), f2_mul(y, sn)), qh[ks][r], ql[ks][r]);
          f2_split_bf16(f2_fma(y, c, f2_mul(x, sn)), qh[ks + KS / 2][r], ql[ks + KS / 2][r]);
        }
      }
      // ---- S = q K^T over kvr keys (n-tiles of 8)
      float s[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        if (nt * 8 < kvr) {
          const int krow = nt * 8 + (lane & 7);
#pragma unroll
          for (int k2 = 0; k2 < D / 32; ++k2) {
            uint32_t bb[4];
            ldsm_x4(kaddr(b, krow, k2 * 4 + (lane >> 3)), bb);
            mma_16816(s[nt], qh[2 * k2], bb[0], bb[1]);
            mma_16816(s[nt], qh[2 * k2 + 1], bb[2], bb[3]);
            mma_16816(s[nt], ql[2 * k2], bb[0], bb[1]);
            mma_16816(s[nt], ql[2 * k2 + 1], bb[2], bb[3]);
          }
        }
      }
      // ---- softmax over the NK valid keys (rows: lane/4 and lane/4 + 8)
      float ma = kNegInf, mb = kNegInf;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        if (nt * 8 + 8 > NK) {  // the n-tile holding the last key, or past it (uniform)
          const int key = nt * 8 + 2 * (lane & 3);
          s[nt][0] = key < NK ? s[nt][0] : kNegInf;
          s[nt][1] = key + 1 < NK ? s[nt][1] : kNegInf;
          s[nt][2] = key < NK ? s[nt][2] : kNegInf;
          s[nt][3] = key + 1 < NK ? s[nt][3] : kNegInf;
        }
        ma = max3f(ma, s[nt][0], s[nt][1]);
        mb = max3f(mb, s[nt][2], s[nt][3]);
      }
      ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
      ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
      float la = 0.f, lb = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        if (nt * 8 < kvr) {
          s[nt][0] = ex2_approx(s[nt][0] - ma);
          s[nt][1] = ex2_approx(s[nt][1] - ma);
          la += s[nt][0] + s[nt][1];
          if (G8) {
            s[nt][2] = s[nt][3] = 0.f;
          } else {
            s[nt][2] = ex2_approx(s[nt][2] - mb);
            s[nt][3] = ex2_approx(s[nt][3] - mb);
            lb += s[nt][2] + s[nt][3];
          }
        }
      }
      la += __shfl_xor_sync(0xffffffffu, la, 1);
      la += __shfl_xor_sync(0xffffffffu, la, 2);
      lb += __shfl_xor_sync(0xffffffffu, lb, 1);
      lb += __shfl_xor_sync(0xffffffffu, lb, 2);
      // ---- O = P V: key steps of 16, then one of 8 when kvr is an odd multiple of 8
      float o[D / 8][4];
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        if (kk * 16 + 16 <= kvr) {
          uint32_t pa[4];
          pa[0] = float2_to_bf16x2(s[2 * kk][0], s[2 * kk][1]);
          pa[1] = float2_to_bf16x2(s[2 * kk][2], s[2 * kk][3]);
          pa[2] = float2_to_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
          pa[3] = float2_to_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
          const int vrow = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int dq = 0; dq < D / 16; ++dq) {
            uint32_t bb[4];
            ldsm_x4_trans(vaddr(b, vrow, dq * 2 + (lane >> 4)), bb);
            mma_16816(o[2 * dq], pa, bb[0], bb[1]);
            mma_16816(o[2 * dq + 1], pa, bb[2], bb[3]);
          }
        } else if (kk * 16 + 8 == kvr) {
          const uint32_t a0 = float2_to_bf16x2(s[2 * kk][0], s[2 * kk][1]);
          const uint32_t a1 = float2_to_bf16x2(s[2 * kk][2], s[2 * kk][3]);
          const int vrow = kk * 16 + (lane & 7);
#pragma unroll
          for (int cq = 0; cq < D / 32; ++cq) {  // four 8-column n-tiles per load
            uint32_t bb[4];
            ldsm_x4_trans(vaddr(b, vrow, cq * 4 + (lane >> 3)), bb);
#pragma unroll
            for (int m = 0; m < 4; ++m) mma_1688(o[4 * cq + m], a0, a1, bb[m]);
          }
        }
      }
      // ---- rows 0..G-1 straight to global (row lane/4; rows lane/4 + 8 when G > 8)
      const int ra = lane >> 2, rb = ra + 8;
      const float ia = rcp_approx(la), ib = rcp_approx(lb);
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        const int col = dn * 8 + 2 * (lane & 3);
        if (ra < G)
          *reinterpret_cast<uint32_t*>(out + (int64_t)ra * D + col) = float2_to_bf16x2(o[dn][0] * ia, o[dn][1] * ia);
        if (!G8 && rb < G)
          *reinterpret_cast<uint32_t*>(out + (int64_t)rb * D + col) = float2_to_bf16x2(o[dn][2] * ib, o[dn][3] * ib);
      }
    }
    // buffer b is free for the unit after next; its shared-memory reads and the
    // key rotation's writes come before the tensor copies that refill it
    fence_proxy_async_smem();
    __syncwarp();
    if (!more) break;
    u = un;
    p = pn;
    g = gn;
    un += W;
    pn = un / prm.Hkv;
    gn = un - pn * prm.Hkv;
    bad_cur = bad_next;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int r = 0; r < 4; ++r) qcur[ks][r] = qnext[ks][r];
  }
}

// [rows][d] bf16 viewed as 64-column boxes of box_rows rows, 128-byte swizzle.
int encode_rows(CUtensorMap* m, const void* base, int64_t rows, int d, int box_rows) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return GIST_ATTN_ERR_LAUNCH;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GIST_ATTN_OK : GIST_ATTN_ERR_UNSUPPORTED;
}

// Tensor copies need whole swizzle atoms per cached block (a multiple of 8 rows),
// boxes of at most 256 rows and row coordinates below 2^31.
bool tma_path(const Problem& pb) {
  const int64_t pool_rows = (int64_t)pb.num_blocks * pb.L * 2 * pb.Hkv * pb.block_len;
  return pb.blocks_per_pair > 0 && pb.block_len % 8 == 0 && pb.block_len <= 256 &&
         pool_rows < 0x7fffffff && (int64_t)pb.P * pb.Hkv < 0x7fffffff;
}

template <int D, bool G8, bool TMA>
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
  prm.kvr = (pb.C + 1 + 7) / 8 * 8;
  prm.region = Region<D>::bytes(prm.kvr);
  prm.units = pb.P * pb.Hkv;
  prm.scale_log2 = pb.scale_log2;
  for (int j = 0; j < 64; ++j) prm.theta[j] = pb.inv_freq_d[j];
  alignas(64) CUtensorMap tm_pool{}, tm_kn{}, tm_vn{};
  if (TMA) {
    int rc = encode_rows(&tm_pool, pb.kv_pool, (int64_t)pb.num_blocks * pb.L * 2 * pb.Hkv * pb.block_len,
                         D, pb.block_len);
    if (rc == GIST_ATTN_OK) rc = encode_rows(&tm_kn, pb.k_new, (int64_t)pb.P * pb.Hkv, D, 1);
    if (rc == GIST_ATTN_OK) rc = encode_rows(&tm_vn, pb.v_new, (int64_t)pb.P * pb.Hkv, D, 1);
    if (rc != GIST_ATTN_OK) return rc;
  }
  const uint32_t bytes = kWarps * prm.region;
  if (cudaFuncSetAttribute(decode_short_kernel<D, G8, TMA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_short_kernel<D, G8, TMA>, kThreads,
                                                    bytes) != cudaSuccess ||
      per_sm < 1)
    return GIST_ATTN_ERR_LAUNCH;
  // persistent: one wave of resident CTAs walks all units
  const int64_t need = (prm.units + kWarps - 1) / kWarps;
  const int64_t grid = need < (int64_t)sms * per_sm ? need : (int64_t)sms * per_sm;
  decode_short_kernel<D, G8, TMA><<<(unsigned)grid, kThreads, bytes, stream>>>(prm, tm_pool, tm_kn, tm_vn);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

template <int D, bool G8>
int launch_path(const Problem& pb, cudaStream_t stream) {
  return tma_path(pb) ? launch_d<D, G8, true>(pb, stream) : launch_d<D, G8, false>(pb, stream);
}

}  // namespace

bool decode_short_fits(const Problem& pb) {
  return pb.l == 1 && pb.G <= 16 && pb.C + 1 <= kMaxKeys && pb.blocks_per_pair <= kMaxBlocks &&
         (pb.d == 64 || pb.d == 128) && (int64_t)pb.P * pb.Hkv <= (1 << 30);  // int unit indices
}

int launch_decode_short(const Problem& pb, cudaStream_t stream) {
  const bool g8 = pb.G <= 8;
  if (pb.d == 64) return g8 ? launch_path<64, true>(pb, stream) : launch_path<64, false>(pb, stream);
  if (pb.d == 128) return g8 ? launch_path<128, true>(pb, stream) : launch_path<128, false>(pb, stream);
  return GIST_ATTN_ERR_UNSUPPORTED;
}

}  // namespace gattn
