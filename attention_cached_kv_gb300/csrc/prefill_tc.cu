// prefill_tc.cu -- attention of l >= 2 new tokens against a short cached
// segment on the 5th-generation tensor core (tcgen05, TMEM accumulators).
//
// [Gist page, "在线的一次 attention"]: per pair and layer, K = cat(G_item, K_new),
// V = cat(G_item, V_new), queries numbered after the cached positions, causal
// inside the new block, nothing written back.  [Gist page, "收益有多大：存储"]:
// the Hq/Hkv query heads of a group share one KV head, so a unit of work is
// (pair, KV head) and its rows are (token, head-in-group), token-major, which is
// the memory order of q/out.  [Gist page, "收益有多大：算力"]: only the logits,
// the softmax and softmax x V depend on the KV length; they are this kernel.
//
// Persistent CTAs (two per SM when TMEM and shared memory allow), warp-specialised:
//   * warp 8 (MMA): tcgen05.mma issue (S = Q K^T, O = P V);
//   * warp 9 (TMA): TMA loads of 128-row Q tiles into a 3-stage ring and TMA
//     stores of O, so that waiting for a store never delays the tensor core;
//   * warps 10.. (K/V: one, or three where a unit is a single tile, or four
//     with one CTA per SM): stage each unit's K/V into one of two buffers one
//     unit ahead (cached rows through the pool gather, new rows raw, by 16-byte
//     cp.async; an E4M3 pool's cached rows are dequantised by their block
//     scales on the way in), convert the cached keys to f16 and rotate the new
//     keys in place, and hand the buffer over by an mbarrier; the tensor core's
//     commit after the unit's last P V hands it back.  This keeps the staging
//     off the compute warps, whose per-row work sets the pace;
//   * warps 0-7 (compute): two threads per tile row (TMEM lane = row; the
//     halves split the columns).  They rotate q, run the softmax out of TMEM (P
//     back into TMEM as bf16), and normalise O into the stage for the store.
//   S = q K^T takes q and K in f16: rotated q and the rotated new keys are
//   rounded once to f16 (11 significant bits, where bf16 has 8), and the cached
//   bf16 keys convert to f16 exactly (magnitudes in [2^-17, 65504]).  A key
//   chunk with a value past the f16 range is written as NaN and a rotated q
//   value past it becomes inf, so every row that meets one ends with a
//   non-finite softmax sum and is stored as NaN; the CTA notes that, and once
//   its last store has landed it recomputes those rows in fp32 from the inputs
//   (exact.cuh), so the result holds on the whole bf16 range while the hot
//   loop carries no extra code.  A row whose largest logit passes kExactLogit
//   (where the f16 rounding of q nears the parity bound) is sent there too, by
//   taking +inf for its maximum.  P V stays
//   bf16 x bf16.  Inputs that arrive rotated (the QKV projection's epilogue
//   rotated and rounded them once) skip the rotation and the conversion:
//   S = q K^T runs on the bf16 values as stored.
//   Rotation angles: the base angle pos theta_j of a unit's first token is
//   reduced modulo 2 pi in double (rope_reduce), and token t adds t theta_j in
//   fp32, so positions anywhere in int32 keep their accuracy.
// Hand-offs use mbarriers; the compute warps are software-pipelined so that the
// rotation of tile i+1 runs while O(i) = P V is on the tensor core and the
// normalisation of tile i runs while S(i+1) is.  One pass covers a tile's
// whole key range (up to 288 keys: S in two MMAs past 256 columns), so the
// softmax needs no running rescale.
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
// Two CTAs share an SM for d = 64 with at most 96 keys (three 16-column chunks
// per thread); wider tiles and d = 128 run one CTA per SM.
__host__ __device__ constexpr bool two_per_sm(int D, int NCH) { return D == 64 && NCH <= 4; }
// K/V warps: where two CTAs share an SM, one when a unit spans several tiles
// and three when it is one tile (ℓ ≤ ⌊128/G⌋: the unit's copies and key
// conversion then recur every tile); four where one CTA per SM leaves
// registers for them (d = 128 units carry twice the bytes, wide key sets more rows)
__host__ __device__ constexpr int kv_warps(int D, int NCH) { return two_per_sm(D, NCH) ? 1 : 4; }
constexpr int kKvWarpsOneTile = 3;
// + the MMA warp, the TMA warp and the K/V warps
__host__ __device__ constexpr int threads_of(int KVW) { return kCompute + 64 + 32 * KVW; }
constexpr uint32_t kBarKV = 1;  // named barrier of the K/V warps
constexpr int kMaxStages = 3;  // q/O stages: 3, or 2 where that lets two CTAs share an SM
constexpr int kMaxKeys = 288;  // S, P and O of a 128-row tile within 512 TMEM columns
constexpr int kMaxSmem = 227 * 1024;
constexpr int kMaxBlocksPerPair = 64;

struct TcParams {
  const bf16* k_new;
  const bf16* v_new;
  PoolView pv;
  const int32_t* pos_offset;
  int32_t* status;
  int l, Hkv, G, C;
  int tab_bufs;   // angle tables: 1 (one position layout for every pair), 2 (per unit)
  int tab_rows;   // rows of a table: l, or 16 + ceil(l / 16) for a two-level one
  int Tm;         // tokens per M-tile
  int n_mt;       // M-tiles per unit
  int num_units;  // P * Hkv
  int kv_rows;    // rows of one K (or V) panel
  int rotated;    // q and k_new arrive rotated: no RoPE, S = q K^T in bf16 as stored
  uint32_t stage_bytes, off_kv, kv_buf_bytes, off_tab, tab_stride, off_red, off_bias, off_base,
      off_bar;
  uint32_t p_col, o_col, tmem_cols;  // TMEM plan: S at column 0
  float scale_log2;
  float inv_freq[64];
  ExactInputs ex;  // the inputs again, for rows recomputed in fp32
  bf16* out;
  // FP8 pool: one fp32 scale per (block, layer, K|V, KV head), the pool's rows
  // E4M3 bytes at the same element offsets; null for a bf16 pool
  const float* kv_scale;
};

struct Layout {
  int Tm, n_mt, kv_rows, stages, tab_rows;
  uint32_t stage_bytes, off_kv, kv_buf_bytes, off_tab, tab_stride, off_red, off_bias, off_base,
      off_bar, bytes;
  uint32_t p_col, o_col, tmem_cols;
};

Layout plan_stages(const Problem& pb, int stages) {
  Layout L{};
  L.stages = stages;
  const int np = pb.d / 64;
  L.Tm = 128 / pb.G;
  L.n_mt = (pb.l + L.Tm - 1) / L.Tm;
  L.kv_rows = (pb.C + pb.l + 15) / 16 * 16;  // also the widest S of any tile
  L.stage_bytes = (uint32_t)np * 128 * 128;
  uint32_t off = (uint32_t)stages * L.stage_bytes;
  L.off_kv = off;
  L.kv_buf_bytes = 2u * np * L.kv_rows * 128;  // K panels then V panels
  off += 2 * L.kv_buf_bytes;
  L.off_tab = off;
  // per token: (cos, cos, sin, sin) of frequency pairs, 16 B each, +16 B so that
  // consecutive tokens start on different banks
  L.tab_stride = (uint32_t)(pb.d / 4) * 16 + 16;
  // one table when every pair's new tokens sit at the same positions, else
  // one per K/V buffer (the K/V warp fills the next unit's while the compute
  // warps read the current one's).  Tiles of more than 128 keys (long new
  // blocks) take a two-level table: rows t < 16 hold the angles of tokens
  // 0..15, rows 16 + a those of the offsets 16 a, and a token's angle is the
  // sum of its two (angle addition in the rotation).
  L.tab_rows = L.kv_rows > 96 ? 16 + (pb.l + 15) / 16 : pb.l;
  off += (pb.pos_offset ? 2u : 1u) * (uint32_t)L.tab_rows * L.tab_stride;
  L.off_red = off;
  off += 2u * 2 * 128 * 4;  // partial row max and row sum of each half
  L.off_bias = off;
  off += 17u * 16 * 4;  // mask rows: bias[v][e] = 0 for e < v, else -inf
  L.off_base = off;
  off += (uint32_t)pb.d * 4;  // base angles of a table's first token (set-up; K/V warp)
  L.off_bar = off;
  off += 128;
  L.bytes = off + 1024;
  // TMEM: S [0, N) fp32, P [N, 1.5N) bf16 pairs, O [o, o+d)
  L.p_col = (uint32_t)L.kv_rows;
  L.o_col = (uint32_t)((L.kv_rows * 3 / 2 + 15) / 16 * 16);
  const uint32_t need = L.o_col + pb.d;
  L.tmem_cols = need <= 256 ? 256 : 512;
  return L;
}

// Two CTAs share an SM when d = 64, the TMEM plan is 256 columns and shared
// memory holds two; where three q/O stages miss that by the shared memory, two
// stages take their place.
constexpr uint32_t kTwoPerSmBytes = 113 * 1024;
Layout plan(const Problem& pb) {
  const Layout L3 = plan_stages(pb, kMaxStages);
  if (L3.bytes > (uint32_t)kMaxSmem) return plan_stages(pb, 2);  // wide key sets
  // (wider key sets than 96 run one CTA per SM for their registers anyway)
  if (pb.d == 64 && L3.kv_rows <= 128 && L3.tmem_cols == 256 && L3.bytes > kTwoPerSmBytes) {
    const Layout L2 = plan_stages(pb, 2);
    if (L2.bytes <= kTwoPerSmBytes) return L2;
  }
  return L3;
}

// Rotate one 16-byte chunk of x (elements j0..j0+7) against its partner chunk y
// (elements j0+d/2..): (x, y) <- (x cos - y sin, y cos + x sin), fp32 pairs.
// The table row holds (cos_j, cos_j+1, sin_j, sin_j+1) per frequency pair; a
// second row (two-level tables, else null) adds its angles to the first's.
__device__ __forceinline__ void rope_chunk(const uint4& x, const uint4& y, const uint8_t* trow,
                                           const uint8_t* trow_hi, int j0, uint64_t (&xr)[4],
                                           uint64_t (&yr)[4]) {
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint4 cs = *reinterpret_cast<const uint4*>(trow + ((j0 >> 1) + e) * 16);
    uint64_t c = f2_make(__uint_as_float(cs.x), __uint_as_float(cs.y));
    uint64_t sn = f2_make(__uint_as_float(cs.z), __uint_as_float(cs.w));
    if (trow_hi) {
      const uint4 hs = *reinterpret_cast<const uint4*>(trow_hi + ((j0 >> 1) + e) * 16);
      const uint64_t hc = f2_make(__uint_as_float(hs.x), __uint_as_float(hs.y));
      const uint64_t hsn = f2_make(__uint_as_float(hs.z), __uint_as_float(hs.w));
      const uint64_t c2 = f2_sub(f2_mul(c, hc), f2_mul(sn, hsn));
      sn = f2_fma(sn, hc, f2_mul(c, hsn));
      c = c2;
    }
    const uint64_t xf = bf16x2_to_f2(xw[e]), yf = bf16x2_to_f2(yw[e]);
    xr[e] = f2_sub(f2_mul(xf, c), f2_mul(yf, sn));
    yr[e] = f2_fma(yf, c, f2_mul(xf, sn));
  }
}

// A shared store ordered only against the other volatile shared accesses
// (lds16 / sts16 / barriers), not against plain C++ loads: for stores whose
// target no plain load in the same stretch of code reads.
__device__ __forceinline__ void sts16_ordered(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w));
}

// fp32 pair -> f16 pair, round to nearest even (|x| >= 65520 gives inf)
__device__ __forceinline__ uint32_t f2_to_f16x2(uint64_t v) {
  float a, b;
  f2_split(v, a, b);
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
// bf16 pair -> f16 pair (exact for magnitudes in [2^-17, 65504])
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  return f2_to_f16x2(bf16x2_to_f2(v));
}
// An f16 chunk of eight keys' elements, or all NaN if one of them is not
// finite (past the f16 range): every logit that reads the chunk becomes NaN,
// which sends those rows to the fp32 recomputation.
// Eight E4M3 values (bytes of a, then of b) times `scale`, rounded once to
// f16 (F16) or bf16: one 16-byte chunk of a tile row.
template <bool F16>
__device__ __forceinline__ uint4 e4m3x8_scaled(uint32_t a, uint32_t b, float scale) {
  const uint32_t pr[4] = {a & 0xffffu, a >> 16, b & 0xffffu, b >> 16};
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float lo, hi;
    f16x2_to_floats(e4m3_pair_to_f16x2(pr[e]), lo, hi);
    w[e] = F16 ? f2_to_f16x2(f2_make(lo * scale, hi * scale)) : float2_to_bf16x2(lo * scale, hi * scale);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint4 f16_chunk_or_nan(uint4 h) {
  const uint32_t e = 0x7c007c00u;
  const bool bad = (h.x & 0x7c00u) == 0x7c00u || (h.x & 0x7c000000u) == 0x7c000000u ||
                   (h.y & 0x7c00u) == 0x7c00u || (h.y & 0x7c000000u) == 0x7c000000u ||
                   (h.z & 0x7c00u) == 0x7c00u || (h.z & 0x7c000000u) == 0x7c000000u ||
                   (h.w & 0x7c00u) == 0x7c00u || (h.w & 0x7c000000u) == 0x7c000000u;
  const uint32_t nan2 = e | 0x02000200u;
  return bad ? make_uint4(nan2, nan2, nan2, nan2) : h;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// TMEM load of 16 columns of this thread's lane that also returns their maximum.
// It does not wait: the maximum is valid after tcgen05.wait::ld, which the
// caller issues once for several such loads (ld_red_wait).
__device__ __forceinline__ float ld16_max_async(uint32_t taddr) {
  uint32_t r[16];
  float m;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, %16, [%17];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=f"(m)
      : "r"(taddr));
  return m;
}
// Waits for this thread's TMEM loads; the maxima of the loads pass through it.
template <int N>
__device__ __forceinline__ void ld_red_wait(float (&m)[N]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+f"(m[i]));
}

struct Bars {
  uint64_t qfull[kMaxStages];
  uint64_t rope_done;  // compute -> MMA warp: q tile rotated (hi in the stage, lo in TMEM)
  uint64_t s_done;     // tensor core -> compute: S ready
  uint64_t p_done;     // compute -> MMA warp: P ready
  uint64_t o_done;     // tensor core -> compute: O ready
  uint64_t o_stored[2];  // compute -> TMA warp: O of tile i written into its stage
                         // (two, alternating: the compute warps can finish tile i+1
                         // before the TMA warp has waited on tile i)
  uint64_t kv_ready[2];  // K/V warp -> compute warps: buffer b holds its unit, prepared
  uint64_t kv_free[2];   // tensor core (commit after the unit's last P V) -> K/V warp
  int unit_bad[2];       // buffer b's unit has a block id out of range
  uint64_t drain;  // the MMA warp's last commit: no MMA in flight at teardown
  uint32_t tmem_slot;
  int flagged;  // a row of this CTA came out non-finite (repaired at the end)
};

// NCH: S chunks of 16 columns per thread (the tile's keys / 32, rounded up).
// KVW: K/V warps.  FP8: the pool holds E4M3 bytes and scales.  Registers: each of the 4 SM sub-partitions holds 16 K; two
// CTAs of 11 warps (one K/V warp) put 6 warps on one of them (85 registers a
// thread), of 13 warps (three) 7 (73); one CTA of 14 warps puts 4 (128).
template <int D, int NCH, int NS, int KVW, bool FP8>
__global__ void __launch_bounds__(threads_of(KVW), two_per_sm(D, NCH) ? 2 : 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_o,
                      const __grid_constant__ TcParams prm) {
  constexpr int NP = D / 64;   // 64-column panels
  constexpr int CPR = D / 8;   // 16-byte chunks per row
  constexpr int kThreads = threads_of(KVW);
  constexpr bool TAB2 = NCH > 3;  // two-level angle tables (tiles of more than 96 keys)
  constexpr int KVT = 32 * KVW;  // K/V threads
  constexpr int HALF = D / 2;
  constexpr float kNegInf = -INFINITY;
  constexpr uint32_t kPanel = 128 * 128;  // one 128-row Q panel

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + prm.off_bar);
  float* red_max = reinterpret_cast<float*>(smem + prm.off_red);  // [2][128]
  float* red_sum = red_max + 256;                                  // [2][128]
  float* bias = reinterpret_cast<float*>(smem + prm.off_bias);  // [17][16]
  float* base_ang = reinterpret_cast<float*>(smem + prm.off_base);  // [d/2]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = prm.G, C = prm.C, l = prm.l, Tm = prm.Tm, n_mt = prm.n_mt;
  const uint32_t kv_panel = (uint32_t)prm.kv_rows * 128;
  const int my_units = blockIdx.x < prm.num_units
                           ? (prm.num_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1
                           : 0;
  const int my_tiles = my_units * n_mt;
  auto unit_of = [&](int k) { return (int)blockIdx.x + k * (int)gridDim.x; };
  // tile i uses q/O stage i mod stages, in its (i / stages)-th round
  auto stage_of = [](int i) { return i % NS; };
  auto stage_round = [](int i) { return (uint32_t)(i / NS) & 1u; };

  // ---- set-up (all threads)
  if (warp == 8) {
    tc::tmem_alloc(smem_u32(&bars->tmem_slot), prm.tmem_cols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kMaxStages; ++s) mbar_init(&bars->qfull[s], 1);
    mbar_init(&bars->rope_done, kCompute);
    mbar_init(&bars->s_done, 1);
    mbar_init(&bars->p_done, kCompute);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->o_stored[0], kCompute);
    mbar_init(&bars->o_stored[1], kCompute);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->kv_ready[b], 1);
      mbar_init(&bars->kv_free[b], 1);
    }
    bars->flagged = 0;
    fence_mbar_init();
  }
  {
    const uint4 z = make_uint4(0, 0, 0, 0);
    const int pad = prm.kv_rows - (C + l);  // key rows no copy writes
    for (int idx = tid; idx < 2 * 2 * NP * pad * 8; idx += kThreads) {
      const int c = idx & 7, rr = (idx >> 3) % pad, rest = (idx >> 3) / pad;  // buf, kv, panel
      const uint32_t base = sbase + prm.off_kv + (rest / (2 * NP)) * prm.kv_buf_bytes +
                            ((rest / NP) & 1) * NP * kv_panel + (rest % NP) * kv_panel;
      sts16(base + swz128(C + l + rr, c), z);
    }
    for (int idx = tid; idx < 17 * 16; idx += kThreads) bias[idx] = (idx & 15) < (idx >> 4) ? 0.f : kNegInf;
    const int qpad = 128 - Tm * G;  // rows of each Q stage that no TMA box reaches
    for (int idx = tid; idx < NS * NP * qpad * 8; idx += kThreads) {
      const int c = idx & 7, rr = (idx >> 3) % qpad, sp = (idx >> 3) / qpad;
      sts16(sbase + (sp / NP) * prm.stage_bytes + (sp % NP) * kPanel + swz128(Tm * G + rr, c), z);
    }
  }
  // (cos, sin) of (pos_base + t) theta_j for every new token t < l: the base
  // angle reduced in double by threads j < d/2 (then a barrier), t theta_j in fp32
  auto build_base = [&](int pos_base) {
    if (tid < HALF) base_ang[tid] = rope_reduce(pos_base, prm.ex.theta[tid]);
  };
  // Rows [r0, r1) of a table: a token row t holds (cos, sin) of its base angle
  // ba (reduced in double) plus t theta_j; a two-level table's rows 16 + a
  // hold the angles of 16 a theta_j alone (reduced in double).
  auto fill_rows = [&](uint8_t* table, const float* ba, int r0, int r1, int first, int nthreads) {
    for (int idx = first; idx < (r1 - r0) * (HALF / 2); idx += nthreads) {
      const int row = r0 + idx / (HALF / 2), jp = idx % (HALF / 2);
      float a0, a1;
      if (TAB2 && row >= 16) {
        a0 = rope_reduce(16 * (row - 16), prm.ex.theta[2 * jp]);
        a1 = rope_reduce(16 * (row - 16), prm.ex.theta[2 * jp + 1]);
      } else {
        a0 = fmaf((float)row, prm.inv_freq[2 * jp], ba[2 * jp]);
        a1 = fmaf((float)row, prm.inv_freq[2 * jp + 1], ba[2 * jp + 1]);
      }
      float s0, c0, s1, c1;
      sincosf(a0, &s0, &c0);
      sincosf(a1, &s1, &c1);
      *reinterpret_cast<float4*>(table + row * prm.tab_stride + jp * 16) = make_float4(c0, c1, s0, s1);
    }
  };
  // the angle table of K/V buffer b's unit
  auto table_of = [&](int b) -> uint8_t* {
    return smem + prm.off_tab + (prm.tab_bufs == 2 ? b : 0) * (uint32_t)prm.tab_rows * prm.tab_stride;
  };
  // the table rows of new token t: the token's own (or its offset t mod 16)
  // and, for two-level tables, that of 16 floor(t / 16)
  auto trow_lo = [&](const uint8_t* table, int t) { return table + (TAB2 ? (t & 15) : t) * prm.tab_stride; };
  auto trow_hi = [&](const uint8_t* table, int t) -> const uint8_t* {
    return TAB2 ? table + (16 + (t >> 4)) * prm.tab_stride : nullptr;
  };
  if (!prm.pos_offset) {
    build_base(C);
    __syncthreads();
    fill_rows(table_of(0), base_ang, 0, prm.tab_rows, tid, kThreads);
  } else if (TAB2) {
    // the offset rows of both tables do not depend on the unit's position
    for (int b = 0; b < 2; ++b) fill_rows(table_of(b), base_ang, 16, prm.tab_rows, tid, kThreads);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_slot;

  if (warp == 8) {
    // ================================================================ MMA issue
    // All 32 lanes walk the loop (waits are uniform); lane 0 issues.
    bool failed = false;
    // tile i is the mt-th tile of this CTA's k-th unit (kept incrementally:
    // no integer division on the per-tile path)
    for (int i = 0, k = 0, mt = 0; i < my_tiles; ++i, mt = (mt + 1 == n_mt) ? (++k, 0) : mt + 1) {
      const uint32_t par = (uint32_t)i & 1u;
      const uint32_t stage = sbase + stage_of(i) * prm.stage_bytes;
      const uint32_t kb = sbase + prm.off_kv + (k & 1) * prm.kv_buf_bytes;
      const uint32_t vb = kb + NP * kv_panel;
      const int N = (C + min(l, (mt + 1) * Tm) + 15) & ~15;
      // ---- S = q K^T (f16 x f16, or bf16 x bf16 for inputs that arrive rotated)
      if (__any_sync(0xffffffffu, !mbar_wait(&bars->rope_done, par))) { failed = true; break; }
      tc::fence_after_sync();
      if (lane == 0) {
        // one MMA covers at most 256 keys: wider tiles take a second one for
        // keys 256.. (K rows 256.. start 32 swizzle atoms further on)
        const int N1 = min(N, 256);
        const uint32_t id1 =
            prm.rotated ? tc::idesc_bf16_f32(128, N1, 0) : tc::idesc_f16_f32(128, N1, 0);
        const uint32_t id2 = prm.rotated ? tc::idesc_bf16_f32(128, N > 256 ? N - 256 : 16, 0)
                                         : tc::idesc_f16_f32(128, N > 256 ? N - 256 : 16, 0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t koff = (uint32_t)(ks & 3) * 32;  // 16 columns = 32 bytes
          const uint64_t a = tc::smem_desc_sw128(stage + (ks >> 2) * kPanel + koff, 16, 1024);
          const uint64_t bd = tc::smem_desc_sw128(kb + (ks >> 2) * kv_panel + koff, 16, 1024);
          tc::mma_ss(tmem, a, bd, id1, ks > 0);
          if (N > 256) {
            const uint64_t bd2 = tc::smem_desc_sw128(kb + (ks >> 2) * kv_panel + 256 * 128 + koff, 16, 1024);
            tc::mma_ss(tmem + 256, a, bd2, id2, ks > 0);
          }
        }
        tc::commit(smem_u32(&bars->s_done));
      }
      __syncwarp();
      // ---- O = P V (A = P from TMEM, B = V with d contiguous).  Every compute
      // thread arrives on p_done(i) after reading O(i-1), so O may be overwritten.
      if (__any_sync(0xffffffffu, !mbar_wait(&bars->p_done, par))) { failed = true; break; }
      tc::fence_after_sync();
      if (lane == 0) {
        const uint32_t idesc = tc::idesc_bf16_f32(128, D, 1);
        for (int ks = 0; ks < N / 16; ++ks) {
          const uint64_t bd = tc::smem_desc_sw128(vb + ks * 2048, kv_panel, 1024);
          tc::mma_ts(tmem + prm.o_col, tmem + prm.p_col + ks * 8, bd, idesc, ks > 0);
        }
        tc::commit(smem_u32(&bars->o_done));
        // the unit's last P V: its K/V buffer is free once this completes
        if (mt == n_mt - 1) tc::commit(smem_u32(&bars->kv_free[k & 1]));
      }
      __syncwarp();
    }
    // every MMA this warp issued completes before the CTA tears TMEM down
    // (after a timed-out wait too): one commit, one bounded wait
    if (lane == 0) tc::commit(smem_u32(&bars->drain));
    __syncwarp();
    if (!mbar_wait(&bars->drain, 0)) failed = true;
    if (lane == 0 && failed) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
    __syncwarp();
  } else if (warp == 9) {
    // ================================================================ TMA
    // Q tiles in, O tiles out; a stage is refilled NS tiles on as soon as
    // the store of its output has read it.
    bool failed = false;
    // loads and stores each walk the tiles in order: (unit, tile-in-unit) cursors
    int lk = 0, lmt = 0, sk = 0, smt = 0;
    auto load_tile = [&](int i) {  // i = the next tile to load
      if (i >= my_tiles) return;
      const int u = unit_of(lk), mt = lmt, s = stage_of(i);
      if (++lmt == n_mt) {
        lmt = 0;
        ++lk;
      }
      const int p = u / prm.Hkv, g = u % prm.Hkv;
      mbar_arrive_expect_tx(&bars->qfull[s], (uint32_t)NP * Tm * G * 128);
#pragma unroll
      for (int pn = 0; pn < NP; ++pn)
        tma_load_5d(sbase + s * prm.stage_bytes + pn * kPanel, &tm_q, &bars->qfull[s], 0, pn,
                    g * G, mt * Tm, p);
    };
    if (lane == 0 && my_tiles > 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_o);
      for (int i = 0; i < NS; ++i) load_tile(i);
    }
    int i = 0;  // tiles stored
    for (; i < my_tiles; ++i) {
      if (__any_sync(0xffffffffu, !mbar_wait(&bars->o_stored[i & 1], (uint32_t)(i >> 1) & 1u))) {
        failed = true;
        break;
      }
      if (lane == 0) {
        const int u = unit_of(sk), mt = smt, s = stage_of(i);
        if (++smt == n_mt) {
          smt = 0;
          ++sk;
        }
        const int p = u / prm.Hkv, g = u % prm.Hkv;
#pragma unroll
        for (int pn = 0; pn < NP; ++pn)
          tma_store_5d(&tm_o, sbase + s * prm.stage_bytes + pn * kPanel, 0, pn, g * G, mt * Tm, p);
        bulk_commit();
        bulk_wait_read_all();
        load_tile(i + NS);
      }
      __syncwarp();
    }
    if (lane == 0) {
      bulk_wait_all();
      fence_proxy_async_global();  // the stores are visible to the repair step
      if (failed) {
        report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
        // q loads issued for tiles i .. i + NS - 1 land before the CTA leaves
        for (int t = i; t < i + NS && t < my_tiles; ++t) mbar_wait(&bars->qfull[stage_of(t)], stage_round(t));
      }
    }
    __syncwarp();
  } else if (warp >= 10) {
    // ================================================================ K/V
    // Unit k goes to buffer k & 1 once the tensor core has finished unit k - 2
    // there: cp.async of its rows (cached through the pool gather, new ones
    // raw), then the cached keys converted to f16 and the new keys rotated at
    // the unit's positions and rounded once to f16, in place (a chunk past the
    // f16 range becomes NaN, which sends the rows that read it to the fp32
    // recomputation).  Inputs that arrive rotated are only copied.
    auto chunk_addr = [](uint32_t base, uint32_t pstride, int row, int J) {
      return base + (J >> 3) * pstride + swz128(row, J & 7);
    };
    const int bl = prm.pv.block_len, bpp = prm.pv.blocks_per_pair;
    const size_t row_stride = (size_t)prm.Hkv * D;  // between consecutive new tokens
    const int kt = tid - (kCompute + 64);           // K/V thread index
    auto kv_sync = [&]() {
      if (KVT == 32) __syncwarp(); else named_bar_sync(kBarKV, KVT);
    };
    bool failed = false;
    for (int k = 0; k < my_units && !failed; ++k) {
      const int b = k & 1, u = unit_of(k), p = u / prm.Hkv, g = u - p * prm.Hkv;
      if (k >= 2 && !mbar_wait(&bars->kv_free[b], (uint32_t)((k >> 1) - 1) & 1u)) failed = true;
      if (KVT == 32 ? __any_sync(0xffffffffu, failed) : named_bar_or(kBarKV, KVT, failed)) {
        failed = true;
        break;
      }
      const uint32_t kb = sbase + prm.off_kv + b * prm.kv_buf_bytes;
      const uint32_t vb = kb + NP * kv_panel;
      bool bad = false;
      for (int bi = 0; bi < bpp; ++bi) {
        const int32_t blk = pool_block_id(prm.pv, p, bi);  // the same in every lane
        if (!pool_block_ok(prm.pv, blk)) {
          bad = true;
          continue;
        }
        const bf16* ks = pool_row(prm.pv, blk, g, 0, 0);
        const bf16* vs = pool_row(prm.pv, blk, g, 1, 0);
        if constexpr (FP8) {
          // FP8 pool: 16 E4M3 bytes of a row at a time, dequantised by the
          // block's scales straight into the tiles (keys to f16 with chunks past
          // its range NaN, or bf16 for inputs that arrive rotated; values to
          // bf16), with their own loads: the block is a few rows
          const uint8_t* base8 = reinterpret_cast<const uint8_t*>(prm.pv.pool);
          const uint8_t* k8 = base8 + (ks - prm.pv.pool);
          const uint8_t* v8 = base8 + (vs - prm.pv.pool);
          const int64_t si = (((int64_t)blk * prm.pv.num_layers + prm.pv.layer) * 2) * prm.Hkv + g;
          const float ksc = prm.kv_scale[si], vsc = prm.kv_scale[si + prm.Hkv];
          for (int w = kt; w < bl * (D / 16); w += KVT) {
            const int t = w / (D / 16), c = 2 * (w % (D / 16));  // f16 chunks c, c + 1
            const uint4 kr = __ldg(reinterpret_cast<const uint4*>(k8 + t * D + c * 8));
            const uint4 vr = __ldg(reinterpret_cast<const uint4*>(v8 + t * D + c * 8));
            const int row = bi * bl + t;
            if (prm.rotated) {
              sts16(chunk_addr(kb, kv_panel, row, c), e4m3x8_scaled<false>(kr.x, kr.y, ksc));
              sts16(chunk_addr(kb, kv_panel, row, c + 1), e4m3x8_scaled<false>(kr.z, kr.w, ksc));
            } else {
              sts16(chunk_addr(kb, kv_panel, row, c), f16_chunk_or_nan(e4m3x8_scaled<true>(kr.x, kr.y, ksc)));
              sts16(chunk_addr(kb, kv_panel, row, c + 1),
                    f16_chunk_or_nan(e4m3x8_scaled<true>(kr.z, kr.w, ksc)));
            }
            sts16(chunk_addr(vb, kv_panel, row, c), e4m3x8_scaled<false>(vr.x, vr.y, vsc));
            sts16(chunk_addr(vb, kv_panel, row, c + 1), e4m3x8_scaled<false>(vr.z, vr.w, vsc));
          }
        } else {
          for (int w = kt; w < bl * CPR; w += KVT) {
            const int t = w / CPR, c = w % CPR;
            const uint32_t o = (c >> 3) * kv_panel + swz128(bi * bl + t, c & 7);
            cp_async16(kb + o, ks + t * D + c * 8);
            cp_async16(vb + o, vs + t * D + c * 8);
          }
        }
      }
      const bf16* kn = prm.k_new + ((size_t)p * l * prm.Hkv + g) * D;
      const bf16* vn = prm.v_new + ((size_t)p * l * prm.Hkv + g) * D;
      for (int w = kt; w < l * CPR; w += KVT) {
        const int t = w / CPR, c = w % CPR;
        cp_async16(chunk_addr(kb, kv_panel, C + t, c), kn + t * row_stride + c * 8);
        cp_async16(chunk_addr(vb, kv_panel, C + t, c), vn + t * row_stride + c * 8);
      }
      cp_async_commit();
      uint8_t* table = table_of(b);
      if (prm.pos_offset && !prm.rotated) {
        // this unit's angle table (the compute warps read it for q as well)
        if (kt < HALF) base_ang[HALF + kt] = rope_reduce(prm.pos_offset[p], prm.ex.theta[kt]);
        if (KVT < HALF && kt + KVT < HALF)
          base_ang[HALF + kt + KVT] = rope_reduce(prm.pos_offset[p], prm.ex.theta[kt + KVT]);
        kv_sync();
        fill_rows(table, base_ang + HALF, 0, TAB2 ? 16 : l, kt, KVT);
      }
      cp_async_wait_all();
      kv_sync();  // every K/V thread's copies (and table rows) have landed
      if (!bad && !prm.rotated) {
        for (int bi = 0; bi < (FP8 ? 0 : bpp); ++bi) {  // (an FP8 pool's keys are f16 already)
          for (int w = kt; w < bl * CPR; w += KVT) {
            const int t = w / CPR, c = w % CPR;
            const uint32_t a = chunk_addr(kb, kv_panel, bi * bl + t, c);
            const uint4 v = lds16(a);
            sts16(a, f16_chunk_or_nan(make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y),
                                                 bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w))));
          }
        }
        for (int w = kt; w < l * (CPR / 2); w += KVT) {
          const int t = w / (CPR / 2), J = w % (CPR / 2);
          const uint32_t a0 = chunk_addr(kb, kv_panel, C + t, J);
          const uint32_t a1 = chunk_addr(kb, kv_panel, C + t, J + CPR / 2);
          uint64_t xr[4], yr[4];
          rope_chunk(lds16(a0), lds16(a1), trow_lo(table, t), trow_hi(table, t), 8 * J, xr, yr);
          sts16(a0, f16_chunk_or_nan(make_uint4(f2_to_f16x2(xr[0]), f2_to_f16x2(xr[1]),
                                                f2_to_f16x2(xr[2]), f2_to_f16x2(xr[3]))));
          sts16(a1, f16_chunk_or_nan(make_uint4(f2_to_f16x2(yr[0]), f2_to_f16x2(yr[1]),
                                                f2_to_f16x2(yr[2]), f2_to_f16x2(yr[3]))));
        }
      }
      if (kt == 0) {
        bars->unit_bad[b] = bad ? 1 : 0;
        if (bad) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
      }
      fence_proxy_async_smem();  // the tensor core reads K/V next
      kv_sync();
      if (kt == 0) mbar_arrive(&bars->kv_ready[b]);
    }
    if (failed && kt == 0) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
    cp_async_wait_all();
  } else {
    // ================================================================ compute
    const int h = warp >> 2;               // which half of the row's columns
    const int r = (warp & 3) * 32 + lane;  // tile row == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    auto chunk_addr = [](uint32_t base, uint32_t pstride, int row, int J) {
      return base + (J >> 3) * pstride + swz128(row, J & 7);
    };
    // A wait that has timed out once turns every later wait of this thread
    // into a no-op, so a stuck pipeline ends in bounded time (the status word
    // says so); the loop structure and every barrier stay uniform.
    bool failed = false;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (!failed && !mbar_wait(bar, parity)) failed = true;
    };
    const uint32_t pair_bar = 2 + (warp & 3);  // this row's two threads (warps w, w + 4)
    const int row_tok = r / G;                  // token of row r within its tile
    // Rotate row r of tile i's q (this half's chunk pairs) into the stage as f16.
    // Rows past the tile's tokens hold zeros (TMA fill, or set-up for rows no
    // box reaches), so they come out zero without a select.
    auto rope_tile = [&](int i, int mt, const uint8_t* tab) {
      const int s = stage_of(i);
      const uint32_t stage = sbase + s * prm.stage_bytes;
      const int t0 = mt * Tm, toks = min(Tm, l - t0);
      const int tt = min(row_tok, toks - 1);
      wait(&bars->qfull[s], stage_round(i));
      // q that arrives rotated stays in the stage as loaded (bf16).  A warp whose
      // 32 rows are all past the tile's tokens skips the work: rows are
      // independent in both products, and such rows are never stored.
      if (prm.rotated || (warp & 3) * 32 >= toks * G) {
        tc::fence_before_sync();
        mbar_arrive(&bars->rope_done);
        return;
      }
      constexpr int JH = CPR / 4;  // chunk pairs per half
      const uint8_t* trow = trow_lo(tab, t0 + tt);
      const uint8_t* trh = trow_hi(tab, t0 + tt);
      // All of this thread's chunks are read before the first store, and the
      // stores leave the table reads free to move, so one shared-memory round
      // trip covers the whole row half.
      uint4 xs[JH], ys[JH];
#pragma unroll
      for (int jj = 0; jj < JH; ++jj) {
        xs[jj] = lds16(chunk_addr(stage, kPanel, r, h * JH + jj));
        ys[jj] = lds16(chunk_addr(stage, kPanel, r, h * JH + jj + CPR / 2));
      }
#pragma unroll
      for (int jj = 0; jj < JH; ++jj) {
        const int J = h * JH + jj;
        uint64_t xr[4], yr[4];
        rope_chunk(xs[jj], ys[jj], trow, trh, 8 * J, xr, yr);
        sts16_ordered(chunk_addr(stage, kPanel, r, J),
                      make_uint4(f2_to_f16x2(xr[0]), f2_to_f16x2(xr[1]), f2_to_f16x2(xr[2]),
                                 f2_to_f16x2(xr[3])));
        sts16_ordered(chunk_addr(stage, kPanel, r, J + CPR / 2),
                      make_uint4(f2_to_f16x2(yr[0]), f2_to_f16x2(yr[1]), f2_to_f16x2(yr[2]),
                                 f2_to_f16x2(yr[3])));
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      mbar_arrive(&bars->rope_done);
    };

    // unit k's K/V buffer is ready: k-th use of buffer k & 1
    bool bad_unit = false;  // the current unit has a block id out of range
    auto unit_ready = [&](int k) -> bool {
      wait(&bars->kv_ready[k & 1], (uint32_t)(k >> 1) & 1u);
      return bars->unit_bad[k & 1] != 0;
    };
    bool bad_next = false;
    if (my_units > 0) {
      bad_unit = unit_ready(0);
      rope_tile(0, 0, table_of(0));
    }
    for (int i = 0, k = 0, mt = 0; i < my_tiles; ++i, mt = (mt + 1 == n_mt) ? (++k, 0) : mt + 1) {
      const uint32_t par = (uint32_t)i & 1u;
      if (mt == 0 && i > 0) bad_unit = bad_next;
      const bool bad = bad_unit;
      const int t0 = mt * Tm, toks = min(Tm, l - t0);
      const bool valid = row_tok < toks;
      const bool wlive = (warp & 3) * 32 < toks * G;  // warp-uniform, same for the row's partner
      const int tt = min(row_tok, toks - 1);
      const int N = (C + t0 + toks + 15) & ~15;
      // ---- softmax of row r over this half's 16-column chunks c = h, h+2, ...
      // (read from TMEM twice: for the max, then for the exponentials; holding
      // the chunks in registers between the two costs more in spills)
      wait(&bars->s_done, par);
      tc::fence_after_sync();
      const int lim = C + t0 + tt + 1;  // keys row r sees
      const int lim_all = C + t0 + 1;   // keys every row of the tile sees
      // In the exponential pass, chunks c < cd lie below the causal diagonal
      // for every row of the tile; chunks from cd on reach it and take an
      // additive 0 / -inf row from the bias table.  Those run in a separate
      // (not unrolled) loop, so the mask code is not predicated onto the others.
      const int cd = lim_all >> 4;
      const int c_diag = cd + ((cd ^ h) & 1);  // this half's first chunk at the diagonal
      // the row of the bias table for chunk c: 0 for the keys row r sees, -inf after
      auto bias_row = [&](int c) {
        return reinterpret_cast<const float4*>(bias + min(max(lim - c * 16, 0), 16) * 16);
      };
      if (wlive) {
        // The row maximum runs over all N columns, the causally masked ones
        // (later tokens of the tile, zero padding) included: m is at least the
        // maximum over the keys the row sees, so its weights are at most 1 and
        // the result is the same softmax.  Only a masked logit ~100 (log2
        // units) above every visible one could underflow the weights; the sum
        // check below sends such a row to the fp32 recomputation.
        // (the half's loads issued together, one wait for all of them)
        float mxs[NCH];
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) {
          const int c = 2 * cc + h;
          mxs[cc] = c * 16 < N ? ld16_max_async(tmem + lane_base + c * 16) : kNegInf;
        }
        ld_red_wait(mxs);
        float mx0 = mxs[0];
#pragma unroll
        for (int cc = 1; cc < NCH; ++cc) mx0 = fmaxf(mx0, mxs[cc]);
        // A row whose largest logit passes kExactLogit (q.K in f16 too coarse
        // there) takes m = +inf: every weight is 0, the sum too, and the row
        // goes to the fp32 recomputation.
        if (mx0 * prm.scale_log2 > kExactLogit && !prm.rotated) mx0 = INFINITY;
        red_max[h * 128 + r] = mx0;
        named_bar_sync(pair_bar, 64);
        const float m = fmaxf(red_max[r], red_max[128 + r]);
        {
          const float sc = prm.scale_log2;
          const uint64_t sc2 = f2_make(sc, sc), nmc2 = f2_make(-m * sc, -m * sc);
          const uint64_t one2 = f2_make(1.f, 1.f);
          uint64_t acc[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
          // exponentials of chunk c; at the diagonal the bias row joins the offset
          auto exp16 = [&](int c, const uint32_t (&v)[16], const float4* bt) {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              uint64_t off = nmc2;
              if (bt) {
                const float4 bq = bt[e >> 1];
                off = f2_add(nmc2, (e & 1) ? f2_make(bq.z, bq.w) : f2_make(bq.x, bq.y));
              }
              float a, bb;
              f2_split(f2_fma(f2_make(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sc2, off),
                       a, bb);
              const uint64_t pp = f2_make(ex2_approx(a), ex2_approx(bb));
              acc[e & 1] = f2_fma(pp, one2, acc[e & 1]);
              pk[e] = f2_to_bf16x2(pp);
            }
            tc::st8(tmem + lane_base + prm.p_col + c * 8, pk);
          };
#pragma unroll
          for (int cc = 0; cc < NCH; ++cc) {
            const int c = 2 * cc + h;
            if (c < cd && c * 16 < N) {
              uint32_t v[16];
              tc::ld16(tmem + lane_base + c * 16, v);
              tc::wait_ld();
              exp16(c, v, nullptr);
            }
          }
#pragma unroll 1
          for (int c = c_diag; c * 16 < N; c += 2) {
            uint32_t v[16];
            tc::ld16(tmem + lane_base + c * 16, v);
            tc::wait_ld();
            exp16(c, v, bias_row(c));
          }
          float a0, a1, b0, b1;
          f2_split(acc[0], a0, a1);
          f2_split(acc[1], b0, b1);
          red_sum[h * 128 + r] = (a0 + a1) + (b0 + b1);
        }
      }
      tc::wait_st();
      tc::fence_before_sync();
      mbar_arrive(&bars->p_done);
      // ---- next tile's K/V and q rotation (overlaps O = P V on the tensor core)
      if (i + 1 < my_tiles) {
        const bool opens = mt + 1 == n_mt;  // the next tile opens unit k+1
        if (opens) bad_next = unit_ready(k + 1);
        rope_tile(i + 1, opens ? 0 : mt + 1, table_of(opens ? (k + 1) & 1 : k & 1));
      }
      // ---- O of row r, this half's columns, normalised into the stage
      wait(&bars->o_done, par);
      tc::fence_after_sync();
      if (wlive) {
        named_bar_sync(pair_bar, 64);  // the partner's row sum is written
        const uint32_t stage = sbase + stage_of(i) * prm.stage_bytes;
        constexpr int OC = D / 32;  // 16-column chunks per half
        if (bad) {
          if (valid) {
#pragma unroll
            for (int J = 0; J < 2 * OC; ++J)
              sts16(chunk_addr(stage, kPanel, r, h * 2 * OC + J), make_uint4(0, 0, 0, 0));
          }
        } else {
          const float sum = red_sum[r] + red_sum[128 + r];
          const bool fin = sum <= 3.0e38f && sum >= 1.0e-30f;
          const float inv = fin ? rcp_approx(sum) : __int_as_float(0x7fc00000);  // NaN row
          if (valid && !fin) bars->flagged = 1;
          const uint64_t inv2 = f2_make(inv, inv);
#pragma unroll
          for (int c = 0; c < OC; ++c) {
            uint32_t ov[16];
            tc::ld16(tmem + lane_base + prm.o_col + (h * OC + c) * 16, ov);
            tc::wait_ld();
            if (valid) {  // (one 16-column chunk at a time keeps registers low)
              uint32_t w[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                w[e] = f2_to_bf16x2(
                    f2_mul(f2_make(__uint_as_float(ov[2 * e]), __uint_as_float(ov[2 * e + 1])), inv2));
              const int J = (h * OC + c) * 2;
              sts16(chunk_addr(stage, kPanel, r, J), make_uint4(w[0], w[1], w[2], w[3]));
              sts16(chunk_addr(stage, kPanel, r, J + 1), make_uint4(w[4], w[5], w[6], w[7]));
            }
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
    tc::tmem_dealloc(tmem, prm.tmem_cols);
  }
  // rows stored as NaN (a value past the f16 range reached them): recompute in fp32
  if (bars->flagged) {
    for (int k = 0; k < my_units; ++k) {
      const int u = unit_of(k), p = u / prm.Hkv;
      exact_repair_rows<D>(prm.ex, prm.out, p, u - p * prm.Hkv, 0, l, tid, kThreads, prm.status);
    }
  }
}

int encode_map(CUtensorMap* m, const void* base, const Problem& pb, int Tm) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return GIST_ATTN_ERR_LAUNCH;
  const cuuint64_t dims[5] = {64, (cuuint64_t)(pb.d / 64), (cuuint64_t)pb.Hq, (cuuint64_t)pb.l,
                              (cuuint64_t)pb.P};
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

template <int D, int NCH, int NS, int KVW = kv_warps(D, NCH)>
int launch_d(const Problem& pb, const float* kv_scale, cudaStream_t stream) {
  constexpr bool F = false;
  const Layout L = plan(pb);
  if (L.stages != NS) return GIST_ATTN_ERR_UNSUPPORTED;  // shared memory is sized for L.stages
  TcParams prm{};
  prm.k_new = static_cast<const bf16*>(pb.k_new);
  prm.v_new = static_cast<const bf16*>(pb.v_new);
  prm.pv = PoolView{static_cast<const bf16*>(pb.kv_pool), pb.item_ids, pb.block_table,
                    pb.blocks_per_pair, pb.block_len, pb.num_blocks, pb.L, pb.layer, pb.Hkv, pb.d};
  prm.pos_offset = pb.pos_offset;
  prm.status = pb.status;
  prm.l = pb.l;
  prm.Hkv = pb.Hkv;
  prm.G = pb.G;
  prm.C = pb.C;
  prm.tab_bufs = pb.pos_offset ? 2 : 1;
  prm.tab_rows = L.tab_rows;
  prm.Tm = L.Tm;
  prm.n_mt = L.n_mt;
  prm.num_units = pb.P * pb.Hkv;
  prm.kv_rows = L.kv_rows;
  prm.rotated = (pb.flags & GIST_ATTN_FLAG_PREROTATED) ? 1 : 0;
  prm.stage_bytes = L.stage_bytes;
  prm.off_kv = L.off_kv;
  prm.kv_buf_bytes = L.kv_buf_bytes;
  prm.off_tab = L.off_tab;
  prm.tab_stride = L.tab_stride;
  prm.off_red = L.off_red;
  prm.off_bias = L.off_bias;
  prm.off_base = L.off_base;
  prm.off_bar = L.off_bar;
  prm.p_col = L.p_col;
  prm.o_col = L.o_col;
  prm.tmem_cols = L.tmem_cols;
  prm.scale_log2 = pb.scale_log2;
  for (int j = 0; j < 64; ++j) prm.inv_freq[j] = pb.inv_freq[j];
  exact_inputs_from(prm.ex, pb);
  prm.ex.kv_scale = kv_scale;
  prm.out = static_cast<bf16*>(pb.out);
  prm.kv_scale = kv_scale;

  alignas(64) CUtensorMap tm_q, tm_o;
  int rc = encode_map(&tm_q, pb.q, pb, L.Tm);
  if (rc != GIST_ATTN_OK) return rc;
  rc = encode_map(&tm_o, pb.out, pb, L.Tm);
  if (rc != GIST_ATTN_OK) return rc;
  auto kern = kv_scale ? prefill_tc_kernel<D, NCH, NS, KVW, true> : prefill_tc_kernel<D, NCH, NS, KVW, F>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.bytes) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  // Two CTAs per SM only when both fit: two 256-column TMEM allocations and
  // shared memory for two.  A larger TMEM plan or shared memory means one.
  const int per_sm = (two_per_sm(D, NCH) && L.tmem_cols == 256 && L.bytes <= kTwoPerSmBytes) ? 2 : 1;
  const int64_t units = (int64_t)pb.P * pb.Hkv;
  const int grid = (int)(units < (int64_t)sms * per_sm ? units : (int64_t)sms * per_sm);
  kern<<<grid, threads_of(KVW), L.bytes, stream>>>(tm_q, tm_o, prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

}  // namespace

bool prefill_tc_fits(const Problem& pb) {
  if (pb.l < 2 || pb.G > 128 || pb.C + pb.l > kMaxKeys) return false;
  if (pb.blocks_per_pair > kMaxBlocksPerPair) return false;
  if (pb.d != 64 && pb.d != 128) return false;
  if ((int64_t)pb.P * pb.Hkv > 0x7fffffff) return false;
  const Layout L = plan(pb);
  if (L.o_col + pb.d > 512) return false;  // S, P and O within the SM's TMEM
  if (pb.d == 128 && L.kv_rows > 128) return false;  // (built for at most 4 chunks per thread)
  return L.bytes <= (uint32_t)kMaxSmem;
}

namespace {
int launch_any(const Problem& pb, const float* kv_scale, cudaStream_t stream) {
  const Layout L = plan(pb);
  const int chunks = (L.kv_rows / 16 + 1) / 2;  // per thread: chunks h, h+2, ...
  const bool s2 = L.stages == 2;
  const float* ks = kv_scale;
  if (pb.d == 64) {
    constexpr int K3 = kKvWarpsOneTile;
    const bool one = L.n_mt == 1;
    if (chunks <= 2) return one ? launch_d<64, 2, 3, K3>(pb, ks, stream) : launch_d<64, 2, 3>(pb, ks, stream);
    if (chunks <= 3) {
      if (s2) return one ? launch_d<64, 3, 2, K3>(pb, ks, stream) : launch_d<64, 3, 2>(pb, ks, stream);
      return one ? launch_d<64, 3, 3, K3>(pb, ks, stream) : launch_d<64, 3, 3>(pb, ks, stream);
    }
    if (chunks <= 4) return s2 ? launch_d<64, 4, 2>(pb, ks, stream) : launch_d<64, 4, 3>(pb, ks, stream);
    if (chunks <= 6) return s2 ? launch_d<64, 6, 2>(pb, ks, stream) : launch_d<64, 6, 3>(pb, ks, stream);
    return s2 ? launch_d<64, 9, 2>(pb, ks, stream) : launch_d<64, 9, 3>(pb, ks, stream);
  }
  if (pb.d == 128) {  // (two q stages where a per-unit angle table takes the room of a third)
    if (chunks <= 2) return s2 ? launch_d<128, 2, 2>(pb, ks, stream) : launch_d<128, 2, 3>(pb, ks, stream);
    if (chunks <= 3) return s2 ? launch_d<128, 3, 2>(pb, ks, stream) : launch_d<128, 3, 3>(pb, ks, stream);
    return s2 ? launch_d<128, 4, 2>(pb, ks, stream) : launch_d<128, 4, 3>(pb, ks, stream);
  }
  return GIST_ATTN_ERR_UNSUPPORTED;
}

}  // namespace

int launch_prefill_tc(const Problem& pb, cudaStream_t stream) { return launch_any(pb, nullptr, stream); }

// The E4M3 pool: the K/V warps dequantise the cached rows by their scales.
int launch_prefill_tc_fp8(const Problem& pb, const float* kv_scale, cudaStream_t stream) {
  return launch_any(pb, kv_scale, stream);
}

}  // namespace gattn
