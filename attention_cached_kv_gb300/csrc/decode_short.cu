// decode_short.cu -- one new token (l = 1) against a short cached segment:
// the query-gisted relevance step.
//
// [Gist page, "能不能再进一步"]: with the query compressed too, only the EOS
// token is new; it attends to the k item-gist and k' query-gist positions (two
// read-only blocks) and to its own key, and its K/V are never stored.
// [KV page, "Reusable-state"]: o_t = softmax(q_t K_{<=t}^T / sqrt(d_k)) V_{<=t}.
//
// A unit is (pair, KV head): G <= 16 query heads against C <= 32 cached keys and
// the new key.  The cached part runs transposed, S^T = K q^T on mma.sync
// m16n8k16: the keys are the 16 rows of an MMA tile and the query heads its
// 8-wide N (one tile of heads for G <= 8, two for G <= 16), so the 7 heads of a
// 14/2 model leave one column idle instead of nine rows.  The softmax runs down
// the key rows of the accumulator (shuffles across the 8 lanes of a column);
// movmatrix.trans turns P^T into the A layout of O = P V.  The new key (the
// 17th key of the query-gisted workload) meets the unrotated query: the same
// rotation of both cancels in their dot product, so its logits come from one
// more tensor-core pass over the raw bf16 fragments (exact products, fp32
// sum), and the new value joins in fp32 in the epilogue.  The query's B
// fragments come from its rows in shared memory by ldmatrix, are rotated in
// fp32, pre-scaled to log2 units and split into bf16 hi + lo (two MMA passes),
// so the rounding of rotated q stays out of the logits; keys, values and P V
// stay bf16 with fp32 accumulation, so every bf16 input is in range.  The
// output rows go from the accumulators straight to global memory.
//
// Persistent warps, two units in flight per warp: while a warp computes unit n
// from one of its two shared-memory buffers, the tensor copies of unit n + 1
// (its cached K and V blocks as whole {64, block_len} boxes of the pool, one
// lane per block, and its q rows, new key and new value from three more lanes,
// all issued side by side) fill the other buffer and complete on that
// buffer's mbarrier; the block ids of unit n + 2 are on their way.  A wait that
// runs out (1 s) reports GIST_ATTN_STATUS_TIMEOUT, waits once more for the copy
// still in flight and ends the warp.
//
// FP8 pool ([Suffix page, §2 and the end of §5]: 1-byte KV elements, one fp32
// scale per (block, layer, K|V, KV head)): the E4M3 boxes land in the buffer's
// staging rows and are widened to f16 in one pair of swizzled tiles that both
// buffers share (cvt e4m3x2 -> f16x2, exact); the
// query is scaled into the f16 range by a power of two per head and split into
// f16 hi + lo; the K scale multiplies the fp32 logits; each block's V scale
// over the unit's largest multiplies the fp32 weights before they are rounded
// to f16 (so no weight drops into f16's subnormal range because of a small
// scale), and the unit's largest V scale multiplies the output.
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上";
//        [Suffix page] icman.com.cn news 64898;
//        [KV page] "为什么自回归推理缓存 KV，而不缓存历史 Q？".
#include <math.h>

#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace gattn {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxCached = 32;  // two 16-key tiles
constexpr int kMaxBlocks = 32;  // a unit's block ids are held one per lane

struct ShortParams {
  const bf16* q;
  const bf16* k_new;
  const bf16* v_new;
  bf16* out;
  const float* kv_scale;  // FP8: [num_blocks][L][2][Hkv]
  PoolView pv;            // the pool (bf16, or E4M3 bytes at the same element offsets)
  const int32_t* pos_offset;
  int32_t* status;
  int Hq, Hkv, G, C;
  int units;        // P * Hkv (at most 2^30)
  uint32_t region;  // bytes of one warp's shared memory
  float scale_log2;
  double theta[64];  // RoPE frequencies (angles reduced in double)
};

// One warp's shared memory: the swizzled K and V tiles (MT x 16 rows of 128
// bytes per 64-column panel, 128-byte swizzle, 1 KiB-aligned) and the parts of
// two buffers, then the small parts of both buffers, the (cos, sin) table of
// the query's position and the buffers' mbarriers.  With a bf16 pool each
// buffer has its own K and V tiles, which the tensor copies fill; with an FP8
// pool the two buffers share one pair, into which the unit being computed
// widens the E4M3 rows its buffer staged (the copies of the next unit land in
// the other buffer's staging rows meanwhile).  A buffer's own part is the q
// tile (GN x 8 rows per panel, same swizzle) and, FP8, the staged E4M3 rows of
// K and V; its small parts are the new key and value rows.  Keeping the small
// parts out of the 1 KiB-aligned tiles, and the FP8 pool's widened tiles
// single, lets five CTAs of four warps share an SM on the query-gisted shape
// with either pool.
template <int D, int GN, int MT, bool FP8>
struct Region {
  static constexpr int NP = D / 64;
  static constexpr uint32_t kv_panel = MT * 16 * 128;
  static constexpr uint32_t q_panel = GN * 8 * 128;
  static constexpr uint32_t kv_tiles = 2 * NP * kv_panel;          // a K and a V tile
  static constexpr uint32_t own = (FP8 ? 0 : kv_tiles) + NP * q_panel + (FP8 ? 2 * MT * 16 * D : 0);
  static constexpr uint32_t buf = (own + 1023) / 1024 * 1024;      // one buffer's own part
  static constexpr uint32_t buf0 = FP8 ? kv_tiles : 0;              // where buffer 0's part starts
  static constexpr uint32_t kv_step = FP8 ? 0 : buf;                // K/V tiles of buffer 1 - buffer 0
  static constexpr uint32_t q_in = FP8 ? 0 : kv_tiles;              // q tile within a buffer's part
  static constexpr uint32_t small = 2 * D * 2;  // the new key row, then the new value row
  static constexpr uint32_t kn_off = buf0 + 2 * buf;  // buffer b: + b x small
  static constexpr uint32_t vn_off = kn_off + D * 2;
  static constexpr uint32_t tab_off = kn_off + 2 * small;  // float2 [D / 2]
  static constexpr uint32_t bar_off = tab_off + D * 4;
  static constexpr uint32_t bytes = (bar_off + 16 + 1023) / 1024 * 1024;
  // offsets of buffer b's K tile, V tile, q tile and staged E4M3 K and V rows
  static constexpr uint32_t k_at(int b) { return b * kv_step; }
  static constexpr uint32_t v_at(int b) { return b * kv_step + NP * kv_panel; }
  static constexpr uint32_t q_at(int b) { return buf0 + b * buf + q_in; }
  static constexpr uint32_t k8_at(int b) { return q_at(b) + NP * q_panel; }
  static constexpr uint32_t v8_at(int b) { return k8_at(b) + MT * 16 * D; }
};
static_assert(Region<64, 1, 1, false>::bytes == 11 * 1024 && Region<64, 1, 1, true>::bytes == 11 * 1024,
              "the query-gisted shape fits five CTAs of four warps per SM with either pool");

// D: head dim.  GN: 8-head tiles of the N dimension.  MT: 16-key tiles.
template <int D, int GN, int MT, bool FP8>
__global__ void __launch_bounds__(kThreads) decode_short_kernel(const __grid_constant__ ShortParams prm,
                                                                const __grid_constant__ CUtensorMap tm_pool,
                                                                const __grid_constant__ CUtensorMap tm_q,
                                                                const __grid_constant__ CUtensorMap tm_kn,
                                                                const __grid_constant__ CUtensorMap tm_vn) {
  using R = Region<D, GN, MT, FP8>;
  constexpr int NP = D / 64;
  constexpr int CPR = D / 8;  // 16-byte chunks per bf16 row
  constexpr int KS = D / 16;  // k-steps over d
  constexpr float kNegInf = -INFINITY;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int G = prm.G, C = prm.C;
  const int bpp = prm.pv.blocks_per_pair, bl = prm.pv.block_len;
  const int NG = prm.Hkv;  // units per pair
  const int W = gridDim.x * kWarps;
  int u = blockIdx.x * kWarps + warp;
  if (u >= prm.units) return;  // warp-uniform; nothing below synchronises the CTA
  uint8_t* reg = smem + warp * prm.region;
  const uint32_t base = smem_u32(reg);
  // (c_j, s_j, c_j+1, s_j+1) x softmax scale at index j / 2 for even j
  const float4* tab = reinterpret_cast<const float4*>(reg + R::tab_off);
  float2* tabw = reinterpret_cast<float2*>(reg + R::tab_off);
  uint64_t* kvbar = reinterpret_cast<uint64_t*>(reg + R::bar_off);
  if ((base & 1023u) != 0) {  // the swizzle atoms need 1 KiB alignment: never expected
    if (lane == 0) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
    return;
  }
  if (lane == 0) {
    mbar_init(&kvbar[0], 1);
    mbar_init(&kvbar[1], 1);
    fence_mbar_init();
  }
  // rows no copy writes stay zero in both buffers: key rows C.. of the K and V
  // tiles, head rows G.. of the q tile
  const int krows = C;
  for (int b = 0; b < 2; ++b) {
    const int kpad = MT * 16 - krows;
    for (int idx = lane; idx < NP * kpad * 8; idx += 32) {
      const int c = idx & 7, rest = idx >> 3, row = krows + rest % kpad, pn = rest / kpad;
      sts16(base + R::k_at(b) + pn * R::kv_panel + swz128(row, c), make_uint4(0, 0, 0, 0));
      sts16(base + R::v_at(b) + pn * R::kv_panel + swz128(row, c), make_uint4(0, 0, 0, 0));
    }
    for (int idx = lane; idx < NP * GN * 8 * 8; idx += 32) {
      const int c = idx & 7, row = (idx >> 3) % (GN * 8), pn = (idx >> 3) / (GN * 8);
      if (row >= G) sts16(base + R::q_at(b) + pn * R::q_panel + swz128(row, c), make_uint4(0, 0, 0, 0));
    }
  }
  fence_proxy_async_smem();
  __syncwarp();

  // This lane's key rows 16 mt + g8 + 8 hh: live (a cached key) and, FP8, the
  // block whose scales they take -- fixed for the launch.
  bool live[MT][2];
  int kblk[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int row = mt * 16 + g8 + 8 * hh;
      live[mt][hh] = row < krows;
      kblk[mt][hh] = min(row, krows - 1) / bl;
    }

  // (cos, sin) x scale of the query's position, frequency j = lane (and lane +
  // 32): the angle reduced in double
  auto build_tab = [&](int pos) {
    __syncwarp();  // the previous unit's reads are done
#pragma unroll
    for (int e = 0; e < D / 64; ++e) {
      const int j = lane + 32 * e;
      float s, c;
      sincosf(rope_reduce(pos, prm.theta[j]), &s, &c);
      tabw[j] = make_float2(c * prm.scale_log2, s * prm.scale_log2);
    }
    __syncwarp();
  };
  // this lane's angles, frequencies 16 ks + 8 r + 2 t4 (+ 1) at [2 ks + r]: read
  // once per launch where every query sits at the same position
  float4 cs[KS];
  auto load_cs = [&]() {
#pragma unroll
    for (int ks = 0; ks < KS / 2; ++ks)
#pragma unroll
      for (int r = 0; r < 2; ++r) cs[2 * ks + r] = tab[(16 * ks + 8 * r + 2 * t4) >> 1];
  };
  const bool fixed_pos = prm.pos_offset == nullptr;
  if (fixed_pos) {
    build_tab(C);
    load_cs();
  }

  // Per unit, lane b < bpp holds the b-th block id (and, FP8, its K and V scales).
  struct Ids {
    int32_t id;
    float ks, vs;
  };
  auto load_ids = [&](int v, int pv_, int gv) -> Ids {
    Ids r{0, 1.f, 1.f};
    if (v < prm.units && lane < bpp) {
      r.id = pool_block_id(prm.pv, pv_, lane);
      if constexpr (FP8) {
        if (pool_block_ok(prm.pv, r.id)) {
          const int64_t si = (((int64_t)r.id * prm.pv.num_layers + prm.pv.layer) * 2) * prm.Hkv + gv;
          r.ks = prm.kv_scale[si];
          r.vs = prm.kv_scale[si + prm.Hkv];
        }
      }
    }
    return r;
  };
  // Tensor copies of unit (p, KV head g0) into buffer b, issued by the lanes
  // side by side: lane t < bpp copies block t's K and V rows, lanes 29, 30 and
  // 31 the q rows, the new key and the new value.  Lane 0 first sets the
  // barrier's byte count with its one arrival, so copies landing before that
  // cannot complete the phase.  Returns (warp-uniform) whether one of the
  // unit's block ids is out of range, in which case no cached rows are copied.
  auto issue = [&](int p, int g0, int b, int32_t id) -> bool {
    const bool bad = __any_sync(0xffffffffu, lane < bpp && !pool_block_ok(prm.pv, id));
    constexpr uint32_t kv_row_bytes = FP8 ? D : D * 2;
    if (lane == 0) {
      mbar_arrive_expect_tx(&kvbar[b], (bad ? 0u : (uint32_t)(bpp * 2 * bl) * kv_row_bytes) +
                                           (uint32_t)G * D * 2 + 2u * D * 2);
    }
    if (lane < bpp && !bad) {
      const int row_k = (int)((((int64_t)id * prm.pv.num_layers + prm.pv.layer) * 2 * prm.Hkv + g0) * bl);
      const int row_v = row_k + prm.Hkv * bl;
      if constexpr (FP8) {
        tma_load_2d(base + R::k8_at(b) + lane * bl * D, &tm_pool, &kvbar[b], 0, row_k);
        tma_load_2d(base + R::v8_at(b) + lane * bl * D, &tm_pool, &kvbar[b], 0, row_v);
      } else {
#pragma unroll
        for (int x = 0; x < NP; ++x) {
          tma_load_2d(base + R::k_at(b) + x * R::kv_panel + lane * bl * 128, &tm_pool, &kvbar[b], 64 * x,
                      row_k);
          tma_load_2d(base + R::v_at(b) + x * R::kv_panel + lane * bl * 128, &tm_pool, &kvbar[b], 64 * x,
                      row_v);
        }
      }
    }
    if (lane >= 29) {
      if (lane == 29) {
#pragma unroll
        for (int x = 0; x < NP; ++x)
          tma_load_2d(base + R::q_at(b) + x * R::q_panel, &tm_q, &kvbar[b], 64 * x, p * prm.Hq + g0 * G);
      } else {
        const bool k = lane == 30;
        tma_load_2d(base + (k ? R::kn_off : R::vn_off) + b * R::small, k ? &tm_kn : &tm_vn, &kvbar[b], 0,
                    p * prm.Hkv + g0);
      }
    }
    return bad;
  };

  // ---- the walk over units u, u + W, ...: (pair, unit-in-pair) by carries
  const int dp = W / NG, dg = W - dp * NG;
  int p = u / NG, gg = u - p * NG;
  auto step = [&](int& pp, int& gq) {
    gq += dg;
    pp += dp;
    if (gq >= NG) {
      gq -= NG;
      ++pp;
    }
  };
  Ids ids_cur = load_ids(u, p, gg);
  bool bad_cur = issue(p, gg, 0, ids_cur.id);
  int un = u + W, pn = p, gn = gg;
  step(pn, gn);
  Ids ids_next = load_ids(un, pn, gn);

  for (int n = 0;; ++n) {
    const int b = n & 1;
    const uint32_t kt = base + R::k_at(b), vt = base + R::v_at(b), qt = base + R::q_at(b);
    // ---- unit un's copies into the other buffer (free since the last unit),
    // and the block ids of the unit after it
    const bool more = un < prm.units;
    int pa2 = pn, ga2 = gn;
    step(pa2, ga2);
    bool bad_next = false;
    Ids ids_after = ids_next;
    if (more) {
      bad_next = issue(pn, gn, b ^ 1, ids_next.id);
      ids_after = load_ids(un + W, pa2, ga2);
    }
    // unit u's copies are the ((n / 2) + 1)-th phase of its buffer's barrier
    if (__any_sync(0xffffffffu, !mbar_wait(&kvbar[b], (uint32_t)(n >> 1) & 1u))) {
      // give up: report, wait (bounded) for the copy still in flight, stop
      if (lane == 0) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
      if (more) mbar_wait(&kvbar[b ^ 1], (uint32_t)((n + 1) >> 1) & 1u);
      return;
    }

    const int g0 = gg;
    if (bad_cur) {
      bf16* out = prm.out + ((size_t)p * prm.Hq + (size_t)g0 * G) * D;
      for (int idx = lane; idx < G * CPR; idx += 32)
        *reinterpret_cast<uint4*>(out + idx * 8) = make_uint4(0, 0, 0, 0);
      if (lane == 0) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
    } else {
      if (!fixed_pos) {
        build_tab(prm.pos_offset[p]);
        load_cs();
      }
      float vmax = 1.f, vinv = 1.f;  // FP8: the unit's largest V scale and its inverse
      if constexpr (FP8) {
        // widen the E4M3 rows of K and V to f16 in the swizzled tiles
        constexpr int PER = 32 / CPR;  // rows per pass of the warp
        const int c = lane % CPR;
        for (int row = lane / CPR; row < krows; row += PER) {
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const uint2 raw = lds64(base + (kv ? R::v8_at(b) : R::k8_at(b)) + row * D + c * 8);
            sts16((kv ? vt : kt) + (c >> 3) * R::kv_panel + swz128(row, c & 7),
                  make_uint4(e4m3x2_to_f16x2(raw.x & 0xffffu), e4m3x2_to_f16x2(raw.x >> 16),
                             e4m3x2_to_f16x2(raw.y & 0xffffu), e4m3x2_to_f16x2(raw.y >> 16)));
          }
        }
        vmax = lane < bpp ? ids_cur.vs : 0.f;
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, s));
        vinv = vmax > 0.f ? 1.f / vmax : 0.f;
        __syncwarp();
      }

      // ---- q: B fragments of head slot 8 hn + g8 (rotated, scaled, split into
      // hi + lo), and the new key's logits from the unrotated values (the same
      // rotation of q and of the new key cancels in their dot product), on the
      // tensor core: A = the new key in all 16 rows, B = the raw bf16 query, so
      // every row of the result holds the same logits and each lane finds those
      // of its own columns, head slots 8 hn + 2 t4 (+ 1), in sn[hn][0 .. 1].
      // bf16 x bf16 products are exact; the sum is fp32.
      uint32_t qh[GN][KS][2], ql[GN][KS][2];
      float qf[GN];        // FP8: 2^e, the factor the head's f16 query was divided by
      float sn[GN][4];     // logits of the new key (log2 units once scaled)
      uint32_t ka[KS][2];  // A registers a0 (= a1) and a2 (= a3) of k-step ks
      {
        const uint32_t kn = base + R::kn_off + b * R::small;  // the new key
        const int mat = lane >> 3;  // ldmatrix: matrix mat's eight rows all read one chunk
#pragma unroll
        for (int ks = 0; ks < KS; ks += 2) {
          uint32_t r4[4];
          ldsm_x4(kn + (16 * (ks + (mat >> 1)) + 8 * (mat & 1)) * 2, r4);
          ka[ks][0] = r4[0];
          ka[ks][1] = r4[1];
          ka[ks + 1][0] = r4[2];
          ka[ks + 1][1] = r4[3];
        }
      }
#pragma unroll
      for (int hn = 0; hn < GN; ++hn) {
        uint64_t rx[KS], ry[KS];
        uint32_t qr[KS][2];
        q_fragments<D, FP8>(qt, R::q_panel, hn, [&](int ks, int r) { return cs[2 * ks + r]; }, qh[hn],
                            ql[hn], qr, rx, ry, qf[hn]);
        sn[hn][0] = sn[hn][1] = sn[hn][2] = sn[hn][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
          mma16816<false>(sn[hn], ka[ks][0], ka[ks][0], ka[ks][1], ka[ks][1], qr[ks][0], qr[ks][1]);
      }

      // ---- S^T = K q^T: rows = keys 16 mt + g8 (+ 8), columns = head slots 8 hn + 2 t4 (+ 1)
      float s[MT][GN][4], s2[MT][GN][4];  // hi and lo passes in separate chains
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int hn = 0; hn < GN; ++hn)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[mt][hn][e] = s2[mt][hn][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t a[4];
          const int c8 = 2 * ks + (lane >> 4);
          ldsm_x4(kt + (c8 >> 3) * R::kv_panel +
                      swz128(mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, c8 & 7),
                  a);
#pragma unroll
          for (int hn = 0; hn < GN; ++hn) {
            mma16816<FP8>(s[mt][hn], a[0], a[1], a[2], a[3], qh[hn][ks][0], qh[hn][ks][1]);
            mma16816<FP8>(s2[mt][hn], a[0], a[1], a[2], a[3], ql[hn][ks][0], ql[hn][ks][1]);
          }
        }
#pragma unroll
        for (int hn = 0; hn < GN; ++hn)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[mt][hn][e] += s2[mt][hn][e];
      }

      // ---- softmax of every head over its cached keys and the new key
      float pn_[GN][2], il[GN][2];  // weight of the new key and 1 / sum, head slots 8 hn + 2 t4 (+ 1)
      uint32_t pa[MT][4];           // A fragments of P for P V, one per 16-key step
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) pa[mt][0] = pa[mt][1] = pa[mt][2] = pa[mt][3] = 0u;
#pragma unroll
      for (int hn = 0; hn < GN; ++hn) {
        float f0 = 1.f, f1 = 1.f;  // FP8: 2^e of head slots 2 t4, 2 t4 + 1
        if constexpr (FP8) {
          f0 = __shfl_sync(0xffffffffu, qf[hn], 8 * t4);
          f1 = __shfl_sync(0xffffffffu, qf[hn], 8 * t4 + 4);
        }
        float m0 = kNegInf, m1 = kNegInf;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float kf = 1.f;
            if constexpr (FP8) kf = __shfl_sync(0xffffffffu, ids_cur.ks, kblk[mt][hh]);
            float& x0 = s[mt][hn][2 * hh];
            float& x1 = s[mt][hn][2 * hh + 1];
            x0 = live[mt][hh] ? x0 * (kf * f0) : kNegInf;
            x1 = live[mt][hh] ? x1 * (kf * f1) : kNegInf;
            m0 = fmaxf(m0, x0);
            m1 = fmaxf(m1, x1);
          }
        }
#pragma unroll
        for (int sft = 4; sft < 32; sft <<= 1) {
          m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, sft));
          m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, sft));
        }
        const float sn0 = sn[hn][0] * prm.scale_log2;
        const float sn1 = sn[hn][1] * prm.scale_log2;
        m0 = fmaxf(m0, sn0);
        m1 = fmaxf(m1, sn1);
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float e0 = ex2_approx(s[mt][hn][2 * hh] - m0);
            const float e1 = ex2_approx(s[mt][hn][2 * hh + 1] - m1);
            l0 += e0;
            l1 += e1;
            float vf = 1.f;
            if constexpr (FP8) {
              const float vs = __shfl_sync(0xffffffffu, ids_cur.vs, kblk[mt][hh]);
              vf = vs * vinv;
            }
            // P^T rows (keys) -> P rows (head slots): this lane gets head slot
            // 8 hn + g8, keys 16 mt + 8 hh + 2 t4 (+ 1)
            pa[mt][hn + 2 * hh] = movmatrix_trans(pack_p<FP8>(e0 * vf, e1 * vf));
          }
        }
#pragma unroll
        for (int sft = 4; sft < 32; sft <<= 1) {
          l0 += __shfl_xor_sync(0xffffffffu, l0, sft);
          l1 += __shfl_xor_sync(0xffffffffu, l1, sft);
        }
        pn_[hn][0] = ex2_approx(sn0 - m0);
        pn_[hn][1] = ex2_approx(sn1 - m1);
        il[hn][0] = rcp_approx(l0 + pn_[hn][0]);
        il[hn][1] = rcp_approx(l1 + pn_[hn][1]);
      }

      // ---- O = P V: rows = head slots g8 (+ 8), columns 8 dn + 2 t4 (+ 1)
      float o[D / 8][4];
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int dq = 0; dq < D / 16; ++dq) {
          uint32_t bv[4];
          const int c8 = 2 * dq + (lane >> 4);
          ldsm_x4_trans(vt + (c8 >> 3) * R::kv_panel +
                            swz128(mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, c8 & 7),
                        bv);
          mma16816<FP8>(o[2 * dq], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], bv[0], bv[1]);
          mma16816<FP8>(o[2 * dq + 1], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], bv[2], bv[3]);
        }
      }

      // ---- the new value and the normalisation: this lane's rows are head
      // slots 8 hn + g8, whose softmax terms sit in lane g8 / 2 (slot g8 % 2).
      // The rows go straight to global memory (the four lanes of a row write 16
      // contiguous bytes per 8-column step), so no store ever holds a buffer.
#pragma unroll
      for (int hn = 0; hn < GN; ++hn) {
        const int src = g8 >> 1;
        const float pa0 = __shfl_sync(0xffffffffu, pn_[hn][0], src);
        const float pa1 = __shfl_sync(0xffffffffu, pn_[hn][1], src);
        const float ia0 = __shfl_sync(0xffffffffu, il[hn][0], src);
        const float ia1 = __shfl_sync(0xffffffffu, il[hn][1], src);
        const float pnew = (g8 & 1) ? pa1 : pa0, inv = (g8 & 1) ? ia1 : ia0;
        const uint64_t oc = f2_make(vmax * inv, vmax * inv), on = f2_make(pnew * inv, pnew * inv);
        const uint32_t vn = base + R::vn_off + b * R::small;
        const int slot = hn * 8 + g8;
        bf16* orow = prm.out + ((size_t)p * prm.Hq + (size_t)g0 * G + slot) * D;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
          const int col = dn * 8 + 2 * t4;
          const uint64_t r2 = f2_fma(bf16x2_to_f2(lds32(vn + col * 2)), on,
                                     f2_mul(f2_make(o[dn][2 * hn], o[dn][2 * hn + 1]), oc));
          if (slot < G) *reinterpret_cast<uint32_t*>(orow + col) = f2_to_bf16x2(r2);
        }
      }
    }
    // buffer b is free for the unit after next; its shared-memory reads and
    // writes come before the tensor copies that refill it
    fence_proxy_async_smem();
    __syncwarp();
    if (!more) break;
    u = un;
    p = pn;
    gg = gn;
    un += W;
    pn = pa2;
    gn = ga2;
    bad_cur = bad_next;
    ids_cur = ids_next;
    ids_next = ids_after;
  }
}

template <int D, int GN, int MT, bool FP8>
int launch_d(const Problem& pb, const float* kv_scale, cudaStream_t stream) {
  using R = Region<D, GN, MT, FP8>;
  ShortParams prm{};
  prm.q = static_cast<const bf16*>(pb.q);
  prm.k_new = static_cast<const bf16*>(pb.k_new);
  prm.v_new = static_cast<const bf16*>(pb.v_new);
  prm.out = static_cast<bf16*>(pb.out);
  prm.kv_scale = kv_scale;
  prm.pv = PoolView{static_cast<const bf16*>(pb.kv_pool), pb.item_ids, pb.block_table,
                    pb.blocks_per_pair, pb.block_len, pb.num_blocks, pb.L, pb.layer, pb.Hkv, pb.d};
  prm.pos_offset = pb.pos_offset;
  prm.status = pb.status;
  prm.Hq = pb.Hq;
  prm.Hkv = pb.Hkv;
  prm.G = pb.G;
  prm.C = pb.C;
  prm.units = pb.P * pb.Hkv;
  prm.region = R::bytes;
  prm.scale_log2 = pb.scale_log2;
  for (int j = 0; j < 64; ++j) prm.theta[j] = pb.inv_freq_d[j];
  alignas(64) CUtensorMap tm_pool{}, tm_q{}, tm_kn{}, tm_vn{};
  const int64_t pool_rows = (int64_t)pb.num_blocks * pb.L * 2 * pb.Hkv * pb.block_len;
  const int box_rows = pb.block_len;  // a block's rows of one KV head
  int rc = FP8 ? encode_2d(&tm_pool, pb.kv_pool, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pool_rows, D, D,
                           box_rows, false)
               : encode_2d(&tm_pool, pb.kv_pool, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool_rows, D,
                           64, box_rows, true);
  if (rc == GIST_ATTN_OK)
    rc = encode_2d(&tm_q, pb.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (int64_t)pb.P * pb.Hq, D, 64,
                   pb.G, true);
  if (rc == GIST_ATTN_OK)
    rc = encode_2d(&tm_kn, pb.k_new, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (int64_t)pb.P * pb.Hkv, D,
                   D, 1, false);
  if (rc == GIST_ATTN_OK)
    rc = encode_2d(&tm_vn, pb.v_new, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (int64_t)pb.P * pb.Hkv, D,
                   D, 1, false);
  if (rc != GIST_ATTN_OK) return rc;
  const uint32_t bytes = kWarps * R::bytes;
  auto kern = decode_short_kernel<D, GN, MT, FP8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, bytes) != cudaSuccess ||
      per_sm < 1)
    return GIST_ATTN_ERR_LAUNCH;
  // persistent: one wave of resident CTAs walks all units
  const int64_t need = (prm.units + kWarps - 1) / kWarps;
  const int64_t grid = need < (int64_t)sms * per_sm ? need : (int64_t)sms * per_sm;
  kern<<<(unsigned)grid, kThreads, bytes, stream>>>(prm, tm_pool, tm_q, tm_kn, tm_vn);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

template <int D, bool FP8>
int launch_shape(const Problem& pb, const float* kv_scale, cudaStream_t stream) {
  const bool g2 = pb.G > 8, m2 = pb.C > 16;
  if (g2)
    return m2 ? launch_d<D, 2, 2, FP8>(pb, kv_scale, stream) : launch_d<D, 2, 1, FP8>(pb, kv_scale, stream);
  return m2 ? launch_d<D, 1, 2, FP8>(pb, kv_scale, stream) : launch_d<D, 1, 1, FP8>(pb, kv_scale, stream);
}

}  // namespace

// l = 1, 1 <= C <= 32 cached keys in blocks of a multiple of 8 rows (whole
// swizzle atoms per tensor copy), at most 16 query heads per KV head.
bool decode_short_fits(const Problem& pb) {
  const int64_t pool_rows = (int64_t)pb.num_blocks * pb.L * 2 * pb.Hkv * pb.block_len;
  return pb.l == 1 && pb.G <= 16 && pb.C >= 1 && pb.C <= kMaxCached &&
         pb.blocks_per_pair <= kMaxBlocks && pb.block_len % 8 == 0 && pb.block_len <= 256 &&
         (pb.d == 64 || pb.d == 128) && pool_rows < 0x7fffffff &&
         (int64_t)pb.P * pb.Hq < 0x7fffffff && (int64_t)pb.P * pb.Hkv <= (1 << 30);
}

int launch_decode_short(const Problem& pb, cudaStream_t stream) {
  if (pb.d == 64) return launch_shape<64, false>(pb, nullptr, stream);
  if (pb.d == 128) return launch_shape<128, false>(pb, nullptr, stream);
  return GIST_ATTN_ERR_UNSUPPORTED;
}

int launch_decode_short_fp8(const Problem& pb, const float* kv_scale, cudaStream_t stream) {
  if (pb.d == 64) return launch_shape<64, true>(pb, kv_scale, stream);
  if (pb.d == 128) return launch_shape<128, true>(pb, kv_scale, stream);
  return GIST_ATTN_ERR_UNSUPPORTED;
}

}  // namespace gattn
