// prefill_long.cu -- causal attention of long new blocks (l up to thousands of
// tokens) over key sequences streamed by TMA, on the 5th-generation tensor core.
//
// [Gist page, "论文做了什么" and "在线的一次 attention"]: the item is forwarded
// once, offline: [prompt; gist] through every layer, plain causal attention
// over the whole sequence (the gist mask only hides the prompt from tokens
// after the gist, and there are none in this pass); each layer's K/V at the
// gist positions is then stored (gist_kv_store).  Two modes:
//   * q and k_new arrive rotated by the QKV projection's epilogue
//     (GIST_ATTN_FLAG_PREROTATED), no cache: the kernel streams them as stored
//     (bf16 scores);
//   * the staged path (stage.cu): keys and values are a pair's [cached; new]
//     sequence prepared in a workspace, token i sees keys [0, C + i], and the
//     softmax warps rotate q in its stage as it arrives (f16 scores).
//
// A work item is a 128-row tile of one (pair, KV head): floor(128 / G) whole
// tokens x G heads, token-major (the memory order of q/out).  Its keys are the
// keys up to its last token's, in blocks of 128, one pass: per block S = q K^T
// into TMEM, the block's row maxima, P = exp2((S - m) scale) as bf16 into TMEM
// with m the running maximum, O += P V.  m moves only when a block's maximum
// exceeds it by more than 8 (log2 units); then the row's O and sum are scaled
// down first.  P stays below 2^8, the result is exact softmax either way, and O
// is touched in between only for those rare rows: S(b) done means the tensor
// core has finished P V of block b - 1, and P V of block b waits for P.
// Persistent CTAs, two per SM, warp-specialised:
//   * warp 8: streams the K and V blocks by TMA (two slots each) and issues
//     tcgen05.mma (S into TMEM, then O from P in TMEM);
//   * warp 9: TMA loads of the q tiles (two stages) and TMA stores of O;
//   * warps 0-7: two threads per row (TMEM lane = row), the softmax (block
//     maxima by tcgen05.ld.red.max below the causal diagonal, a 0/-inf bias row
//     at it) and the normalisation of O into the stage.
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上".
#include <math.h>

#include "common.cuh"
#include "exact.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace gattn {
namespace {

constexpr int kCompute = 256;            // 8 compute warps
constexpr int kThreads = kCompute + 64;  // + the MMA/K-V warp and the Q/O warp
constexpr int kKB = 128;                 // keys per block
constexpr uint32_t kTile = 128 * 128;    // bytes of a 128-row x 64-column bf16 tile
constexpr int kMaxSmem = 227 * 1024;

struct LongParams {
  int32_t* status;
  int l, Hkv, G, Tm, n_mt, num_tiles;
  int C;    // keys before new token 0 (the staged cache), 0 for whole sequences
  int f16;  // q and keys are f16 (staged), else bf16 as stored
  // q to rotate in the kernel (else null: q arrives rotated): (cos, sin) of
  // pos_offset[p] theta_j [P][32] and of i theta_j [l][32], added per token
  const float2* q_base;
  const float2* q_rel;
  float scale_log2;
  // The call's own inputs: a row whose softmax sum comes out non-finite (an f16
  // key chunk the staged pre-pass wrote as NaN, or a q value past the f16
  // range; with f16 scores also a largest logit past kExactLogit) is stored as
  // NaN and, once the CTA's stores have landed, recomputed from them in fp32
  // (exact.cuh).
  ExactInputs ex;
  bf16* out;
};

// A CTA's tiles are blockIdx.x, blockIdx.x + gridDim.x, ... of the row-major
// (pair, KV head, row tile) order; the walk steps (mt, g, p) by carries, with
// the division done once.
struct TileWalk {
  int dmt, dg, dp;  // gridDim.x split over (row tile, KV head, pair)
  int mt, g, p;     // current tile
  __device__ void init(const LongParams& prm) {
    const int x = (int)blockIdx.x, du = (int)gridDim.x / prm.n_mt;
    dmt = (int)gridDim.x % prm.n_mt;
    dg = du % prm.Hkv;
    dp = du / prm.Hkv;
    mt = x % prm.n_mt;
    const int u = x / prm.n_mt;
    g = u % prm.Hkv;
    p = u / prm.Hkv;
  }
  __device__ void next(const LongParams& prm) {
    mt += dmt;
    int c = 0;
    if (mt >= prm.n_mt) {
      mt -= prm.n_mt;
      c = 1;
    }
    g += dg + c;  // < 2 Hkv
    p += dp;
    if (g >= prm.Hkv) {
      g -= prm.Hkv;
      ++p;
    }
  }
};

// A position in the stream of (tile, key block) steps of one CTA.
struct StepWalk {
  TileWalk t;
  int i, b, nb;  // tile index, block, blocks of the tile
  __device__ static int blocks(const LongParams& prm, int mt) {
    return (prm.C + min(prm.l, (mt + 1) * prm.Tm) + kKB - 1) / kKB;
  }
  __device__ void init(const LongParams& prm) {
    t.init(prm);
    i = b = 0;
    nb = blocks(prm, t.mt);
  }
  __device__ void next(const LongParams& prm) {
    if (++b == nb) {
      b = 0;
      ++i;
      t.next(prm);
      nb = blocks(prm, t.mt);
    }
  }
};

// shared memory: q/O stages [2], K slots [2], V slots [2], then the small parts
constexpr uint32_t kOffQ = 0, kOffK = 2 * kTile, kOffV = 4 * kTile, kOffRed = 6 * kTile;
constexpr uint32_t kOffBias = kOffRed + 3 * 2 * 128 * 4;  // block maxima [2 blocks][2], sums [2]
constexpr uint32_t kOffBar = kOffBias + 17 * 16 * 4;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
// TMEM: S [0, 128) fp32, P [128, 192) bf16 pairs, O [192, 256)
constexpr uint32_t kPCol = 128, kOCol = 192, kTmemCols = 256;

struct LBars {
  uint64_t qfull[2], kfull[2], kfree[2], vfull[2], vfree[2];
  uint64_t s_done, p_done, o_done, o_stored[2];
  uint64_t q_ready[2];  // q rotated in its stage (when it arrives unrotated)
  uint64_t drain;  // the MMA warp's last commit: no MMA in flight at teardown
  uint32_t tmem_slot;
  int flagged;  // a row of this CTA came out non-finite (repaired at the end)
};

// 4-D tiled load into shared memory, completing bytes on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// 32 columns of this thread's lane out of TMEM (completes at tc::wait_ld).
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// TMEM load of 32 columns of this thread's lane that also returns their maximum.
__device__ __forceinline__ float ld32_max(uint32_t taddr) {
  uint32_t r[32];
  float m;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=f"(m)
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+f"(m)::"memory");
  return m;
}

// 16 columns of this thread's lane into TMEM.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// fp32 pair -> f16 pair (round to nearest even), first element in the low half.
__device__ __forceinline__ uint32_t f2_to_f16x2(uint64_t v) {
  float a, b;
  f2_split(v, a, b);
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__global__ void __launch_bounds__(kThreads, 2)
    prefill_long_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_o,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ LongParams prm) {
  constexpr float kNegInf = -INFINITY;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  LBars* bars = reinterpret_cast<LBars*>(smem + kOffBar);
  float* red_max = reinterpret_cast<float*>(smem + kOffRed);  // [2 blocks][2][128]
  float* red_sum = red_max + 512;                              // [2][128]
  float* bias = reinterpret_cast<float*>(smem + kOffBias);     // [17][16]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = prm.G, l = prm.l, Tm = prm.Tm;
  const int my_tiles = (int)blockIdx.x < prm.num_tiles
                           ? (prm.num_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1
                           : 0;

  if (warp == 8) {
    tc::tmem_alloc(smem_u32(&bars->tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->qfull[s], 1);
      mbar_init(&bars->kfull[s], 1);
      mbar_init(&bars->kfree[s], 1);
      mbar_init(&bars->vfull[s], 1);
      mbar_init(&bars->vfree[s], 1);
      mbar_init(&bars->o_stored[s], kCompute);
      mbar_init(&bars->q_ready[s], kCompute);
    }
    mbar_init(&bars->s_done, 1);
    mbar_init(&bars->p_done, kCompute);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->drain, 1);
    bars->flagged = 0;
    fence_mbar_init();
  }
  for (int idx = tid; idx < 17 * 16; idx += kThreads) bias[idx] = (idx & 15) < (idx >> 4) ? 0.f : kNegInf;
  {  // rows of each q stage that no TMA box reaches stay zero
    const int qpad = 128 - Tm * G;
    for (int idx = tid; idx < 2 * qpad * 8; idx += kThreads) {
      const int c = idx & 7, rr = (idx >> 3) % qpad, s = (idx >> 3) / qpad;
      sts16(sbase + kOffQ + s * kTile + swz128(Tm * G + rr, c), make_uint4(0, 0, 0, 0));
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_slot;

  if (warp == 8) {
    // ============================================ K/V blocks by TMA, tcgen05.mma
    // Steps run over this CTA's tiles and their key blocks.  Per step: P V once
    // P is in TMEM, then at once S of the next step (so S done also means the
    // P V before it is done), then the K and V loads two steps ahead, whose
    // slots the S and the P V just issued free.
    bool failed = false;
    int kc = 0, vc = 0, sx = 0, px = 0;  // K, V loads issued; S, P V products issued
    StepWalk kw, vw, sw, pw;             // next K load, V load, S, P V
    kw.init(prm);
    vw.init(prm);
    sw.init(prm);
    pw.init(prm);
    auto load_k = [&]() {
      if (kw.i >= my_tiles) return;
      const int s = kc & 1;
      if (!mbar_wait(&bars->kfree[s], ((uint32_t)(kc >> 1) & 1u) ^ 1u)) failed = true;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->kfull[s], kTile);
        tma_load_4d(sbase + kOffK + s * kTile, &tm_k, &bars->kfull[s], 0, kw.t.g, kw.b * kKB, kw.t.p);
      }
      ++kc;
      kw.next(prm);
    };
    auto load_v = [&]() {
      if (vw.i >= my_tiles) return;
      const int s = vc & 1;
      if (!mbar_wait(&bars->vfree[s], ((uint32_t)(vc >> 1) & 1u) ^ 1u)) failed = true;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->vfull[s], kTile);
        tma_load_4d(sbase + kOffV + s * kTile, &tm_v, &bars->vfull[s], 0, vw.t.g, vw.b * kKB, vw.t.p);
      }
      ++vc;
      vw.next(prm);
    };
    // S = q K^T of the next step into TMEM [0, 128); the compute warps have
    // finished reading the last S (P of its step is done)
    auto issue_s = [&]() {
      if (sw.i >= my_tiles || failed) return;
      const int ks = sx & 1;
      if (__any_sync(0xffffffffu,
                     (sw.b == 0 && !mbar_wait(prm.q_base ? &bars->q_ready[sw.i & 1] : &bars->qfull[sw.i & 1],
                                              (uint32_t)(sw.i >> 1) & 1u)) ||
                         !mbar_wait(&bars->kfull[ks], (uint32_t)(sx >> 1) & 1u))) {
        failed = true;
        return;
      }
      tc::fence_after_sync();
      if (lane == 0) {
        const int kend = prm.C + min(l, (sw.t.mt + 1) * Tm);
        const int N = (min(kKB, kend - sw.b * kKB) + 15) & ~15;
        const uint32_t idesc = prm.f16 ? tc::idesc_f16_f32(128, N, 0) : tc::idesc_bf16_f32(128, N, 0);
        const uint32_t stage = sbase + kOffQ + (sw.i & 1) * kTile;
        const uint32_t kb = sbase + kOffK + ks * kTile;
#pragma unroll
        for (int k16 = 0; k16 < 4; ++k16) {
          const uint64_t a = tc::smem_desc_sw128(stage + k16 * 32, 16, 1024);
          const uint64_t bd = tc::smem_desc_sw128(kb + k16 * 32, 16, 1024);
          tc::mma_ss(tmem, a, bd, idesc, k16 > 0);
        }
        tc::commit(smem_u32(&bars->s_done));
        tc::commit(smem_u32(&bars->kfree[ks]));
      }
      __syncwarp();
      ++sx;
      sw.next(prm);
    };
    if (lane == 0) {
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
    }
    load_k();
    load_k();
    load_v();
    load_v();
    issue_s();
    while (pw.i < my_tiles && !failed) {
      // O (+)= P V once P is in TMEM and V has landed
      const int vs = px & 1;
      if (__any_sync(0xffffffffu, !mbar_wait(&bars->vfull[vs], (uint32_t)(px >> 1) & 1u) ||
                                      !mbar_wait(&bars->p_done, (uint32_t)px & 1u))) {
        failed = true;
        break;
      }
      tc::fence_after_sync();
      if (lane == 0) {
        const int kend = prm.C + min(l, (pw.t.mt + 1) * Tm);
        const int N = (min(kKB, kend - pw.b * kKB) + 15) & ~15;
        const uint32_t idesc = tc::idesc_bf16_f32(128, 64, 1);
        const uint32_t vb = sbase + kOffV + vs * kTile;
        for (int k16 = 0; k16 < N / 16; ++k16) {
          const uint64_t bd = tc::smem_desc_sw128(vb + k16 * 2048, kTile, 1024);
          tc::mma_ts(tmem + kOCol, tmem + kPCol + k16 * 8, bd, idesc, (pw.b > 0 || k16 > 0) ? 1u : 0u);
        }
        tc::commit(smem_u32(&bars->vfree[vs]));
        if (pw.b == pw.nb - 1) tc::commit(smem_u32(&bars->o_done));
      }
      __syncwarp();
      ++px;
      pw.next(prm);
      issue_s();
      load_k();
      load_v();
    }
    // every MMA this warp issued completes before the CTA tears TMEM down
    // (after a timed-out wait too): one commit, one bounded wait
    if (lane == 0) tc::commit(smem_u32(&bars->drain));
    __syncwarp();
    if (!mbar_wait(&bars->drain, 0)) failed = true;
    if (failed && lane == 0) {
      // K and V loads issued and not consumed land before the CTA leaves
      for (int j = sx; j < kc; ++j) mbar_wait(&bars->kfull[j & 1], (uint32_t)(j >> 1) & 1u);
      for (int j = px; j < vc; ++j) mbar_wait(&bars->vfull[j & 1], (uint32_t)(j >> 1) & 1u);
    }
    if (lane == 0 && failed) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
    __syncwarp();
  } else if (warp == 9) {
    // ============================================ q tiles in, O tiles out
    bool failed = false;
    TileWalk qw, ow;  // next q load, next O store
    qw.init(prm);
    ow.init(prm);
    int qi = 0;
    auto load_q = [&]() {
      if (qi >= my_tiles) return;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->qfull[qi & 1], (uint32_t)Tm * G * 128);
        tma_load_5d(sbase + kOffQ + (qi & 1) * kTile, &tm_q, &bars->qfull[qi & 1], 0, 0, qw.g * G,
                    qw.mt * Tm, qw.p);
      }
      ++qi;
      qw.next(prm);
    };
    if (lane == 0 && my_tiles > 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_o);
    }
    load_q();
    load_q();
    int i = 0;  // tiles stored
    for (; i < my_tiles; ++i) {
      if (__any_sync(0xffffffffu, !mbar_wait(&bars->o_stored[i & 1], (uint32_t)(i >> 1) & 1u))) {
        failed = true;
        break;
      }
      if (lane == 0) {
        tma_store_5d(&tm_o, sbase + kOffQ + (i & 1) * kTile, 0, 0, ow.g * G, ow.mt * Tm, ow.p);
        bulk_commit();
        bulk_wait_read_all();
      }
      __syncwarp();
      ow.next(prm);
      load_q();
    }
    if (lane == 0) {
      bulk_wait_all();
      fence_proxy_async_global();  // the stores are visible to the repair step
      if (failed) {
        report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
        // q loads issued for tiles i .. qi - 1 land before the CTA leaves
        for (int t = i; t < qi; ++t) mbar_wait(&bars->qfull[t & 1], (uint32_t)(t >> 1) & 1u);
      }
    }
    __syncwarp();
  } else {
    // ============================================ softmax passes, normalisation
    const int h = warp >> 2;               // which half of the row's columns
    const int r = (warp & 3) * 32 + lane;  // tile row == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t pair_bar = 2 + (warp & 3);
    const int row_tok = r / G;
    bool failed = false;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (!failed && !mbar_wait(bar, parity)) failed = true;
    };
    const float sc = prm.scale_log2;
    // q that arrives unrotated: each thread rotates frequencies [16 h, 16 h + 16)
    // of its row (elements j and j + 32) in the stage and rounds once to f16; the
    // angle is the pair's base plus the token's index angle.  Tile i + 1's q is
    // rotated once tile i's last P is in TMEM, while its P V runs.
    auto rotate_q = [&](int qi, const TileWalk& qt) {
      if (!prm.q_base || qi >= my_tiles) return;
      wait(&bars->qfull[qi & 1], (uint32_t)(qi >> 1) & 1u);
      const int tq = qt.mt * Tm + row_tok;
      if (row_tok < min(Tm, l - qt.mt * Tm) && !failed) {
        const uint32_t stage = sbase + kOffQ + (qi & 1) * kTile;
        const float4* bs = reinterpret_cast<const float4*>(prm.q_base + (size_t)qt.p * 32 + 16 * h);
        const float4* rl = reinterpret_cast<const float4*>(prm.q_rel + (size_t)tq * 32 + 16 * h);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const uint32_t ax = stage + swz128(r, 2 * h + cc), ay = stage + swz128(r, 4 + 2 * h + cc);
          const uint4 xv = lds16(ax), yv = lds16(ay);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, yw[4] = {yv.x, yv.y, yv.z, yv.w};
          uint32_t ox[4], oy[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {  // frequencies 16 h + 8 cc + 2 e, + 1
            const float4 b4 = __ldg(bs + 4 * cc + e), r4 = __ldg(rl + 4 * cc + e);
            const float c0 = b4.x * r4.x - b4.y * r4.y, s0 = b4.y * r4.x + b4.x * r4.y;
            const float c1 = b4.z * r4.z - b4.w * r4.w, s1 = b4.w * r4.z + b4.z * r4.w;
            const float x0 = __uint_as_float(xw[e] << 16), x1 = __uint_as_float(xw[e] & 0xffff0000u);
            const float y0 = __uint_as_float(yw[e] << 16), y1 = __uint_as_float(yw[e] & 0xffff0000u);
            ox[e] = f2_to_f16x2(f2_make(x0 * c0 - y0 * s0, x1 * c1 - y1 * s1));
            oy[e] = f2_to_f16x2(f2_make(y0 * c0 + x0 * s0, y1 * c1 + x1 * s1));
          }
          sts16(ax, make_uint4(ox[0], ox[1], ox[2], ox[3]));
          sts16(ay, make_uint4(oy[0], oy[1], oy[2], oy[3]));
        }
      }
      fence_proxy_async_smem();  // the tensor core reads the stage next
      mbar_arrive(&bars->q_ready[qi & 1]);
    };
    int sx = 0;
    TileWalk tw;
    tw.init(prm);
    rotate_q(0, tw);
    for (int i = 0; i < my_tiles; ++i, tw.next(prm)) {
      const int mt = tw.mt;
      const int nb = StepWalk::blocks(prm, mt);
      const int t0 = mt * Tm, toks = min(Tm, l - t0);
      const bool valid = row_tok < toks;
      const bool wlive = (warp & 3) * 32 < toks * G;  // warp-uniform, same for the row's partner
      const int kend = prm.C + t0 + toks;
      const int lim = prm.C + t0 + min(row_tok, toks - 1) + 1;  // keys row r sees
      const int lim_all = prm.C + t0 + 1;                          // keys every row of the tile sees
      // chunk c (16 keys) of block b: below the diagonal for every row, or at it
      auto bias_row = [&](int key0) {
        return reinterpret_cast<const float4*>(bias + min(max(lim - key0, 0), 16) * 16);
      };
      constexpr float kSlack = 8.f;  // log2 units the running maximum may trail a block's
      const uint64_t sc2 = f2_make(sc, sc);
      const uint64_t one2 = f2_make(1.f, 1.f);
      uint64_t acc[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
      float m = kNegInf;  // running maximum of row r (the same in both threads)
      for (int b = 0; b < nb; ++b) {
        const int N = (min(kKB, kend - b * kKB) + 15) & ~15;
        // S(b) done also means the P V of block b - 1 is done: P and O are quiet
        wait(&bars->s_done, (uint32_t)sx & 1u);
        tc::fence_after_sync();
        if (wlive) {
          // the block's maximum over this half's 32-column groups q = h, h + 2
          // (the second 16 columns of a group may lie past the block's keys)
          float mx = kNegInf;
          for (int q = h; q * 32 < N; q += 2) {
            const int key0 = b * kKB + q * 32;
            const uint32_t ta = tmem + lane_base + q * 32;
            if (key0 + 32 <= lim_all) {
              mx = fmaxf(mx, ld32_max(ta));
            } else {
              uint32_t v[32];
              ld32(ta, v);
              tc::wait_ld();
              const int nh = q * 32 + 16 < N ? 2 : 1;
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                if (hh < nh) {
                  const float4* bt = bias_row(key0 + hh * 16);
#pragma unroll
                  for (int q4 = 0; q4 < 4; ++q4) {
                    const float4 bq = bt[q4];
                    const int o = hh * 16 + 4 * q4;
                    mx = max3f(mx, __uint_as_float(v[o]) + bq.x, __uint_as_float(v[o + 1]) + bq.y);
                    mx = max3f(mx, __uint_as_float(v[o + 2]) + bq.z, __uint_as_float(v[o + 3]) + bq.w);
                  }
                }
              }
            }
          }
          float* slot = red_max + (b & 1) * 256;  // two slots: a partner may still read the last
          slot[h * 128 + r] = mx;
          named_bar_sync(pair_bar, 64);
          const float mb = fmaxf(slot[r], slot[128 + r]);
          // (S - m) scale is in log2 units; the first block always moves m.  A
          // row whose maximum jumps scales its O and sum down first.  The TMEM
          // load and store are warp-collective, so the whole warp takes that
          // branch when any of its rows needs it; the other rows scale by 1.
          const bool move = (mb - m) * sc > kSlack;
          const bool rescale = move && m != kNegInf;
          if (__any_sync(0xffffffffu, rescale)) {
            const float f = rescale ? ex2_approx((m - mb) * sc) : 1.f;
            const uint64_t f2 = f2_make(f, f);
            acc[0] = f2_mul(acc[0], f2);
            acc[1] = f2_mul(acc[1], f2);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t ov[16];
              const uint32_t oa = tmem + lane_base + kOCol + (h * 2 + c) * 16;
              tc::ld16(oa, ov);
              tc::wait_ld();
              uint32_t w[16];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                float x, y;
                f2_split(f2_mul(f2_make(__uint_as_float(ov[2 * e]), __uint_as_float(ov[2 * e + 1])), f2), x, y);
                w[2 * e] = __float_as_uint(x);
                w[2 * e + 1] = __float_as_uint(y);
              }
              tmem_st16(oa, w);
            }
          }
          if (move) m = mb;
          // P = exp2((S - m) scale) into TMEM as bf16 pairs (group q -> P
          // columns [16 q, 16 q + 16)), summed
          const uint64_t nmc2 = f2_make(-m * sc, -m * sc);
          for (int q = h; q * 32 < N; q += 2) {
            const int key0 = b * kKB + q * 32;
            uint32_t v[32];
            ld32(tmem + lane_base + q * 32, v);
            tc::wait_ld();
            const bool two = q * 32 + 16 < N;
            uint32_t pk[16];
            if (key0 + 32 <= lim_all) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                float a, bb;
                f2_split(f2_fma(f2_make(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sc2, nmc2),
                         a, bb);
                const uint64_t pp = f2_make(ex2_approx(a), ex2_approx(bb));
                acc[e & 1] = f2_fma(pp, one2, acc[e & 1]);
                pk[e] = f2_to_bf16x2(pp);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                if (e < 8 || two) {
                  const float4 bq = bias_row(key0 + (e >> 3) * 16)[(e >> 1) & 3];
                  const uint64_t off = f2_add(nmc2, (e & 1) ? f2_make(bq.z, bq.w) : f2_make(bq.x, bq.y));
                  float a, bb;
                  f2_split(f2_fma(f2_make(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sc2, off),
                           a, bb);
                  const uint64_t pp = f2_make(ex2_approx(a), ex2_approx(bb));
                  acc[e & 1] = f2_fma(pp, one2, acc[e & 1]);
                  pk[e] = f2_to_bf16x2(pp);
                }
              }
            }
            const uint32_t pa = tmem + lane_base + kPCol + q * 16;
            if (two) {
              tmem_st16(pa, pk);
            } else {
              tc::st8(pa, *reinterpret_cast<const uint32_t(*)[8]>(pk));
            }
          }
        }
        tc::wait_st();
        tc::fence_before_sync();
        mbar_arrive(&bars->p_done);  // P in TMEM, and S read: the next S may go
        ++sx;
      }
      if (prm.q_base) {  // tile i + 1's q, while this tile's last P V runs
        TileWalk nt = tw;
        nt.next(prm);
        rotate_q(i + 1, nt);
      }
      // ---- O of row r, this half's 32 columns, normalised into the stage
      wait(&bars->o_done, (uint32_t)i & 1u);
      tc::fence_after_sync();
      if (wlive) {
        float a0, a1, b0, b1;
        f2_split(acc[0], a0, a1);
        f2_split(acc[1], b0, b1);
        red_sum[h * 128 + r] = (a0 + a1) + (b0 + b1);
        named_bar_sync(pair_bar, 64);
        const float sum = red_sum[r] + red_sum[128 + r];
        // (f16 scores: a row whose largest logit passes kExactLogit goes to fp32 too)
        const bool fin = sum <= 3.0e38f && !(prm.f16 && m * sc > kExactLogit);
        const float inv = fin ? rcp_approx(sum) : __int_as_float(0x7fc00000);  // NaN row
        if (valid && !fin) bars->flagged = 1;
        const uint32_t stage = sbase + kOffQ + (i & 1) * kTile;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t ov[16];
          tc::ld16(tmem + lane_base + kOCol + (h * 2 + c) * 16, ov);
          tc::wait_ld();
          if (valid) {
            const uint64_t inv2 = f2_make(inv, inv);
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = f2_to_bf16x2(f2_mul(f2_make(__uint_as_float(ov[2 * e]), __uint_as_float(ov[2 * e + 1])), inv2));
            const int J = (h * 2 + c) * 2;
            sts16(stage + swz128(r, J), make_uint4(w[0], w[1], w[2], w[3]));
            sts16(stage + swz128(r, J + 1), make_uint4(w[4], w[5], w[6], w[7]));
          }
        }
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      mbar_arrive(&bars->o_stored[i & 1]);
    }
    if (failed) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 8) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  // rows stored as NaN (a value past the f16 range reached them): recompute in fp32
  if (bars->flagged) {
    TileWalk tw;
    tw.init(prm);
    for (int i = 0; i < my_tiles; ++i, tw.next(prm))
      exact_repair_rows<64>(prm.ex, prm.out, tw.p, tw.g, tw.mt * Tm, min(l, (tw.mt + 1) * Tm), tid,
                            kThreads, prm.status);
  }
}

// q / out: [P][l][Hq][64] as {64, 1, Hq, l, P}, boxes of G heads x Tm tokens
// (2-byte elements, copied as they are).
int encode_qo(CUtensorMap* m, const void* base, const Problem& pb, int Tm) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return GIST_ATTN_ERR_LAUNCH;
  const cuuint64_t dims[5] = {64, 1, (cuuint64_t)pb.Hq, (cuuint64_t)pb.l, (cuuint64_t)pb.P};
  const cuuint64_t strides[4] = {128, (cuuint64_t)pb.d * 2, (cuuint64_t)pb.Hq * pb.d * 2,
                                 (cuuint64_t)pb.l * pb.Hq * pb.d * 2};
  const cuuint32_t box[5] = {64, 1, (cuuint32_t)pb.G, (cuuint32_t)Tm, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GIST_ATTN_OK : GIST_ATTN_ERR_UNSUPPORTED;
}

// keys / values: [P][rows][Hkv][64] as {64, Hkv, rows, P}, boxes of 128 tokens of one head.
int encode_kv(CUtensorMap* m, const void* base, const Problem& pb, int rows) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return GIST_ATTN_ERR_LAUNCH;
  const cuuint64_t dims[4] = {64, (cuuint64_t)pb.Hkv, (cuuint64_t)rows, (cuuint64_t)pb.P};
  const cuuint64_t strides[3] = {(cuuint64_t)pb.d * 2, (cuuint64_t)pb.Hkv * pb.d * 2,
                                 (cuuint64_t)rows * pb.Hkv * pb.d * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)kKB, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GIST_ATTN_OK : GIST_ATTN_ERR_UNSUPPORTED;
}

}  // namespace

// The grid of row tiles fits the kernel's int counters, and its shared memory
// fits a CTA.
bool prefill_long_grid_ok(const Problem& pb, int rows) {
  return pb.d == 64 && pb.G <= 128 && rows > 0 &&
         (int64_t)pb.P * pb.Hkv * ((pb.l + 128 / pb.G - 1) / (128 / pb.G)) < 0x7fffffff &&
         kSmemBytes <= (uint32_t)kMaxSmem;
}

// Pre-rotated inputs, no cached segment, d = 64, groups of at most 128 heads,
// sequences longer than the single-pass kernel's 128 keys.
bool prefill_long_fits(const Problem& pb) {
  return (pb.flags & GIST_ATTN_FLAG_PREROTATED) && pb.C == 0 && pb.l > 128 && prefill_long_grid_ok(pb, pb.l);
}

// q [P][l][Hq][64], keys and values [P][C + l][Hkv][64]: new token i sees keys
// [0, C + i]; q and keys f16 (f16 = true) or bf16.
int launch_prefill_long_on(const Problem& pb, const void* q, const void* k, const void* v, int C,
                           bool f16, const float2* q_base, const float2* q_rel, cudaStream_t stream) {
  LongParams prm{};
  prm.status = pb.status;
  prm.l = pb.l;
  prm.Hkv = pb.Hkv;
  prm.G = pb.G;
  prm.Tm = 128 / pb.G;
  prm.n_mt = (pb.l + prm.Tm - 1) / prm.Tm;
  prm.num_tiles = (int)((int64_t)pb.P * pb.Hkv * prm.n_mt);
  prm.C = C;
  prm.f16 = f16 ? 1 : 0;
  prm.q_base = q_base;
  prm.q_rel = q_rel;
  prm.scale_log2 = pb.scale_log2;
  exact_inputs_from(prm.ex, pb);
  prm.out = static_cast<bf16*>(pb.out);
  alignas(64) CUtensorMap tm_q, tm_o, tm_k, tm_v;
  int rc = encode_qo(&tm_q, q, pb, prm.Tm);
  if (rc == GIST_ATTN_OK) rc = encode_qo(&tm_o, pb.out, pb, prm.Tm);
  if (rc == GIST_ATTN_OK) rc = encode_kv(&tm_k, k, pb, C + pb.l);
  if (rc == GIST_ATTN_OK) rc = encode_kv(&tm_v, v, pb, C + pb.l);
  if (rc != GIST_ATTN_OK) return rc;
  if (cudaFuncSetAttribute(prefill_long_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmemBytes) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  const int grid = prm.num_tiles < 2 * sms ? prm.num_tiles : 2 * sms;
  prefill_long_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tm_q, tm_o, tm_k, tm_v, prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

int launch_prefill_long(const Problem& pb, cudaStream_t stream) {
  return launch_prefill_long_on(pb, pb.q, pb.k_new, pb.v_new, 0, false, nullptr, nullptr, stream);
}

}  // namespace gattn
