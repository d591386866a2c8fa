// prefill.cu -- attention of new tokens against a cached segment of any
// length, streaming the keys: the general path behind the tensor-memory kernel
// (which covers up to 128 keys).  It also runs the offline gist compression's
// causal pass over a whole [prompt; gist] sequence (empty cache, l = j + k).
//
// [Gist page, "在线的一次 attention"]: K = cat(cache[item].K[layer], K_new), V
// likewise; the new tokens are numbered after the cached positions; causal
// inside the new block; nothing is written back.  [Gist page, "论文做了什么"]:
// over [prompt; gist] alone the gist mask is the plain causal mask; with the
// optional per-pair gist start the kernel also applies the full gist mask (a
// token after the gist no longer sees the prompt), the training-layout forward.
//
// One CTA (8 warps) per (pair, KV head, group of whole tokens with at most 128
// rows); rows are (token, head-in-group), token-major -- the memory order of
// q/out, so the group's q rows arrive by one TMA tensor copy per 64-column
// panel (128-byte swizzle) and leave the same way.  Keys stream through a
// double-buffered shared-memory ring in tiles of 64: cached rows by 16-byte
// cp.async through the pool gather (then converted to f16 in place), new values
// by cp.async, new keys rotated in registers on the way in and rounded once to
// f16.  Rotations use angle addition: one table of (cos, sin)(r theta) for
// r < 64 per CTA and a per-tile base angle, so no angle grows with the
// position.  Each warp keeps its 16-row tile's q fragments (rotated, scaled,
// rounded once to f16: 11 significant bits, so the rounding of rotated q stays
// small against the bf16 output), S = q K^T (f16 x f16) and O += P V (bf16 x
// bf16) on mma.sync m16n8k16 with fp32 accumulation, and a running max / sum
// softmax across key tiles.  A key chunk with a value past the f16 range is
// written as NaN and a q value past it becomes inf, so the rows that meet one
// end with a non-finite sum; they, and the rows whose largest logit passes
// kExactLogit, are recomputed in fp32 from the inputs (exact.cuh).  Base angles of a group or key tile are reduced modulo 2 pi in
// double (rope_reduce), so every int32 position keeps its accuracy.
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上".
#include <math.h>

#include "common.cuh"
#include "exact.cuh"
#include "kernels.h"

namespace gattn {
namespace {

constexpr int kThreads = 256;
constexpr int kKT = 64;        // keys per streamed tile
constexpr int kRowsMax = 128;  // rows per CTA (8 warps x 16)
constexpr int kRT = kRowsMax > kKT ? kRowsMax : kKT;  // rows of the (cos, sin)(r theta) table
constexpr int kMaxSmem = 227 * 1024;

struct StreamParams {
  const bf16* k_new;
  const bf16* v_new;
  PoolView pv;
  const int32_t* pos_offset;
  const int32_t* gist_start;  // [P] or nullptr
  int32_t* status;
  int l, Hkv, G, C, gist_len;
  int Tg;        // tokens per CTA
  int ngroups;   // CTAs per (pair, KV head)
  uint32_t off_ring, ring_buf, off_rt, off_bq, off_bk, off_ids, off_bar, q_panel;
  float scale_log2;
  float inv_freq[64];
  ExactInputs ex;  // the inputs again, for rows recomputed in fp32
};

struct Layout {
  int Tg, ngroups;
  uint32_t off_ring, ring_buf, off_rt, off_bq, off_bk, off_ids, off_bar, q_panel, bytes;
};

Layout plan(const Problem& pb) {
  Layout L{};
  const int np = pb.d / 64;
  L.Tg = pb.G >= kRowsMax ? 1 : kRowsMax / pb.G;
  L.ngroups = (pb.l + L.Tg - 1) / L.Tg;
  L.q_panel = kRowsMax * 128;
  uint32_t off = np * L.q_panel;
  L.off_ring = off;
  L.ring_buf = 2u * np * kKT * 128;  // K tile then V tile
  off += 2 * L.ring_buf;
  L.off_rt = off;
  // (cos, sin)(r theta_j) for r < kRT: a key's offset in its tile (< kKT) and a
  // token's offset in its group (< Tg <= kRowsMax)
  off += (uint32_t)kRT * (pb.d / 2) * 8;
  L.off_bq = off;
  off += (uint32_t)(pb.d / 2) * 8;
  L.off_bk = off;
  off += 2u * (pb.d / 2) * 8;  // per ring buffer
  L.off_ids = off;
  off += ((uint32_t)pb.blocks_per_pair * 4 + 15) / 16 * 16;
  L.off_bar = off;
  off += 16;
  L.bytes = off + 1024;
  return L;
}

// fp32 pair -> f16 pair, round to nearest even (|x| >= 65520 gives inf)
__device__ __forceinline__ uint32_t f16pair(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// bf16 pair -> f16 pair (exact for magnitudes in [2^-17, 65504])
__device__ __forceinline__ uint32_t bf16x2_to_f16pair(uint32_t v) {
  return f16pair(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
// An f16 chunk, or all NaN if one element is not finite (past the f16 range):
// the rows whose logits read it then end with a non-finite sum.
__device__ __forceinline__ uint4 f16_chunk_or_nan(uint4 h) {
  const bool bad = (h.x & 0x7c00u) == 0x7c00u || (h.x & 0x7c000000u) == 0x7c000000u ||
                   (h.y & 0x7c00u) == 0x7c00u || (h.y & 0x7c000000u) == 0x7c000000u ||
                   (h.z & 0x7c00u) == 0x7c00u || (h.z & 0x7c000000u) == 0x7c000000u ||
                   (h.w & 0x7c00u) == 0x7c00u || (h.w & 0x7c000000u) == 0x7c000000u;
  const uint32_t nan2 = 0x7e007e00u;
  return bad ? make_uint4(nan2, nan2, nan2, nan2) : h;
}
// D(16x8) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_16816_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (cos, sin) of (base + r) theta from cos/sin of base theta and of r theta.
__device__ __forceinline__ float2 add_angle(float2 b, float2 r) {
  return make_float2(b.x * r.x - b.y * r.y, b.y * r.x + b.x * r.y);
}

template <int D>
__global__ void __launch_bounds__(kThreads, D == 64 ? 2 : 1)
    prefill_stream_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_o,
                          const __grid_constant__ StreamParams prm) {
  constexpr int NP = D / 64;
  constexpr int CPR = D / 8;
  constexpr int HALF = D / 2;
  constexpr float kNegInf = -INFINITY;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sRing = sQ + prm.off_ring;
  const float2* rt = reinterpret_cast<const float2*>(smem + prm.off_rt);  // [kRT][HALF]
  float2* bq = reinterpret_cast<float2*>(smem + prm.off_bq);
  float2* bk = reinterpret_cast<float2*>(smem + prm.off_bk);            // [2][HALF]
  int32_t* ids = reinterpret_cast<int32_t*>(smem + prm.off_ids);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + prm.off_bar);
  const uint32_t kv_panel = kKT * 128;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int unit = blockIdx.x;
  const int grp = unit % prm.ngroups;
  unit /= prm.ngroups;
  const int g = unit % prm.Hkv, p = unit / prm.Hkv;
  const int G = prm.G, C = prm.C, l = prm.l;
  const int t0 = grp * prm.Tg;
  const int Tc = min(prm.Tg, l - t0);
  const int rows = Tc * G;
  const int kmax = C + t0 + Tc;  // keys the group's last token sees
  const int nkt = (kmax + kKT - 1) / kKT;
  const int pos0 = prm.pos_offset ? prm.pos_offset[p] : C;  // position of new token 0

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, (uint32_t)NP * prm.Tg * G * 128);
#pragma unroll
    for (int pn = 0; pn < NP; ++pn) tma_load_5d(sQ + pn * prm.q_panel, &tm_q, bar, 0, pn, g * G, t0, p);
  }
  bool bad = false;
  for (int b = tid; b < prm.pv.blocks_per_pair; b += kThreads) {
    const int32_t blk = pool_block_id(prm.pv, p, b);
    bad |= !pool_block_ok(prm.pv, blk);
    ids[b] = blk;
  }
  for (int idx = tid; idx < kRT * HALF; idx += kThreads) {
    const int r = idx / HALF, j = idx - r * HALF;
    float s, c;
    sincosf((float)r * prm.inv_freq[j], &s, &c);
    reinterpret_cast<float2*>(smem + prm.off_rt)[idx] = make_float2(c, s);
  }
  for (int j = tid; j < HALF; j += kThreads) {
    float s, c;
    sincosf(rope_reduce((long long)pos0 + t0, prm.ex.theta[j]), &s, &c);
    bq[j] = make_float2(c, s);
  }
  bad = __syncthreads_or(bad);

  // tile kt: keys [64 kt, 64 kt + 64) into ring buffer kt & 1
  auto stage = [&](int kt) {
    const uint32_t kb = sRing + (kt & 1) * prm.ring_buf, vb = kb + NP * kv_panel;
    const int k0 = kt * kKT;
    const int inew0 = max(k0 - C, 0);  // first new key of the tile (base of its angles)
    float2* base = bk + (kt & 1) * HALF;
    for (int j = tid; j < HALF; j += kThreads) {
      float s, c;
      sincosf(rope_reduce((long long)pos0 + inew0, prm.ex.theta[j]), &s, &c);
      base[j] = make_float2(c, s);
    }
    __syncthreads();
    for (int idx = tid; idx < kKT * CPR; idx += kThreads) {
      const int r = idx / CPR, c = idx - r * CPR;
      const int kappa = k0 + r;
      const uint32_t ko = (c >> 3) * kv_panel + swz128(r, c & 7);
      if (kappa >= kmax) {
        sts16(kb + ko, make_uint4(0, 0, 0, 0));
        sts16(vb + ko, make_uint4(0, 0, 0, 0));
      } else if (kappa < C) {
        const int b = kappa / prm.pv.block_len, t = kappa - b * prm.pv.block_len;
        cp_async16(kb + ko, pool_row(prm.pv, ids[b], g, 0, t) + c * 8);
        cp_async16(vb + ko, pool_row(prm.pv, ids[b], g, 1, t) + c * 8);
      } else {
        const int i = kappa - C;
        cp_async16(vb + ko, prm.v_new + (((int64_t)p * l + i) * prm.Hkv + g) * D + c * 8);
        if (c < CPR / 2) {  // rotate the pair of chunks (c, c + d/16)
          const bf16* src = prm.k_new + (((int64_t)p * l + i) * prm.Hkv + g) * D;
          const uint4 lo = ldg16(src + c * 8), hi = ldg16(src + HALF + c * 8);
          const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w}, hw[4] = {hi.x, hi.y, hi.z, hi.w};
          uint32_t ol[4], oh[4];
          const int rr = i - inew0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = c * 8 + 2 * e;
            const float2 c0 = add_angle(base[j], rt[rr * HALF + j]);
            const float2 c1 = add_angle(base[j + 1], rt[rr * HALF + j + 1]);
            const float2 x = bf16x2_to_float2(lw[e]), y = bf16x2_to_float2(hw[e]);
            ol[e] = f16pair(x.x * c0.x - y.x * c0.y, x.y * c1.x - y.y * c1.y);
            oh[e] = f16pair(y.x * c0.x + x.x * c0.y, y.y * c1.x + x.y * c1.y);
          }
          sts16(kb + ko, f16_chunk_or_nan(make_uint4(ol[0], ol[1], ol[2], ol[3])));
          const int ch = c + CPR / 2;
          sts16(kb + (ch >> 3) * kv_panel + swz128(r, ch & 7),
                f16_chunk_or_nan(make_uint4(oh[0], oh[1], oh[2], oh[3])));
        }
      }
    }
    cp_async_commit();
  };

  // the cached keys of tile kt (landed, copied by this same thread): bf16 -> f16
  // in place; returns whether the tile had any (then a barrier must follow)
  auto convert_cached = [&](int kt) -> bool {
    const int k0 = kt * kKT;
    if (k0 >= C) return false;
    const uint32_t kb = sRing + (kt & 1) * prm.ring_buf;
    for (int idx = tid; idx < kKT * CPR; idx += kThreads) {
      const int r = idx / CPR, c = idx - r * CPR;
      if (k0 + r < C && k0 + r < kmax) {
        const uint32_t a = kb + (c >> 3) * kv_panel + swz128(r, c & 7);
        const uint4 v = lds16(a);
        sts16(a, f16_chunk_or_nan(make_uint4(bf16x2_to_f16pair(v.x), bf16x2_to_f16pair(v.y),
                                             bf16x2_to_f16pair(v.z), bf16x2_to_f16pair(v.w))));
      }
    }
    return true;
  };

  bool timed_out = !mbar_wait(bar, 0);
  timed_out = __syncthreads_or(timed_out);
  if (timed_out) {
    if (tid == 0) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
    mbar_wait(bar, 0);
    return;
  }

  if (!bad) {
    stage(0);
    cp_async_wait_all();
    if (convert_cached(0)) __syncthreads();
    __syncthreads();
    // ---- this warp's 16-row tile: q fragments rotated, scaled, rounded to f16
    const int r0 = warp * 16;
    const bool active = r0 < rows;
    uint32_t qh[D / 16][4];
    const int ra = r0 + (lane >> 2), rb = ra + 8;
    const int tta = min(ra / G, Tc - 1), ttb = min(rb / G, Tc - 1);
    if (active) {
      const int row = r0 + (lane & 15);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int c8 = ks * 2 + (lane >> 4);
        ldsm_x4(sQ + (c8 >> 3) * prm.q_panel + swz128(row, c8 & 7), qh[ks]);
      }
#pragma unroll
      for (int ks = 0; ks < D / 32; ++ks) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int tt = (r & 1) ? ttb : tta;
          const int j = ks * 16 + 2 * (lane & 3) + ((r & 2) ? 8 : 0);
          const float2 c0 = add_angle(bq[j], rt[tt * HALF + j]);
          const float2 c1 = add_angle(bq[j + 1], rt[tt * HALF + j + 1]);
          const float2 x = bf16x2_to_float2(qh[ks][r]), y = bf16x2_to_float2(qh[ks + D / 32][r]);
          const float sc = prm.scale_log2;
          qh[ks][r] = f16pair((x.x * c0.x - y.x * c0.y) * sc, (x.y * c1.x - y.y * c1.y) * sc);
          qh[ks + D / 32][r] = f16pair((y.x * c0.x + x.x * c0.y) * sc, (y.y * c1.x + x.y * c1.y) * sc);
        }
      }
    }
    // visible keys of a row: [lo, lim); lo > 0 only under the gist mask, for
    // tokens after the gist (their prompt is hidden)
    const int lim_a = C + t0 + tta + 1, lim_b = C + t0 + ttb + 1;
    int lo_a = 0, lo_b = 0;
    if (prm.gist_start) {
      const int gs = max(prm.gist_start[p], 0);
      lo_a = lim_a - 1 >= gs + prm.gist_len ? gs : 0;
      lo_b = lim_b - 1 >= gs + prm.gist_len ? gs : 0;
    }
    float o[D / 8][4];
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
    float m_a = kNegInf, m_b = kNegInf, l_a = 0.f, l_b = 0.f;

    for (int kt = 0; kt < nkt; ++kt) {
      if (kt + 1 < nkt) stage(kt + 1);
      if (active) {
        const uint32_t kb = sRing + (kt & 1) * prm.ring_buf, vb = kb + NP * kv_panel;
        const int k0 = kt * kKT;
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
          const int krow = n * 8 + (lane & 7);
#pragma unroll
          for (int k2 = 0; k2 < D / 32; ++k2) {
            uint32_t b[4];
            const int c8 = k2 * 4 + (lane >> 3);
            ldsm_x4(kb + (c8 >> 3) * kv_panel + swz128(krow, c8 & 7), b);
            mma_16816_f16(s[n], qh[2 * k2], b[0], b[1]);
            mma_16816_f16(s[n], qh[2 * k2 + 1], b[2], b[3]);
          }
        }
        float mx_a = kNegInf, mx_b = kNegInf;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int key = k0 + n * 8 + 2 * (lane & 3);
          s[n][0] = key < lim_a && key >= lo_a ? s[n][0] : kNegInf;
          s[n][1] = key + 1 < lim_a && key + 1 >= lo_a ? s[n][1] : kNegInf;
          s[n][2] = key < lim_b && key >= lo_b ? s[n][2] : kNegInf;
          s[n][3] = key + 1 < lim_b && key + 1 >= lo_b ? s[n][3] : kNegInf;
          mx_a = max3f(mx_a, s[n][0], s[n][1]);
          mx_b = max3f(mx_b, s[n][2], s[n][3]);
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        // a row with no visible key yet keeps max -inf: its weights stay 0
        const float sa = mn_a == kNegInf ? 0.f : mn_a, sb = mn_b == kNegInf ? 0.f : mn_b;
        const float al_a = ex2_approx(m_a - sa), al_b = ex2_approx(m_b - sb);
        m_a = mn_a;
        m_b = mn_b;
        float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          s[n][0] = ex2_approx(s[n][0] - sa);
          s[n][1] = ex2_approx(s[n][1] - sa);
          s[n][2] = ex2_approx(s[n][2] - sb);
          s[n][3] = ex2_approx(s[n][3] - sb);
          sum_a += s[n][0] + s[n][1];
          sum_b += s[n][2] + s[n][3];
        }
        l_a = l_a * al_a + sum_a;
        l_b = l_b * al_b + sum_b;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
          o[dn][0] *= al_a;
          o[dn][1] *= al_a;
          o[dn][2] *= al_b;
          o[dn][3] *= al_b;
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t pa[4];
          pa[0] = float2_to_bf16x2(s[2 * kk][0], s[2 * kk][1]);
          pa[1] = float2_to_bf16x2(s[2 * kk][2], s[2 * kk][3]);
          pa[2] = float2_to_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
          pa[3] = float2_to_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
          const int vrow = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int dq = 0; dq < D / 16; ++dq) {
            uint32_t b[4];
            const int c8 = dq * 2 + (lane >> 4);
            ldsm_x4_trans(vb + (c8 >> 3) * kv_panel + swz128(vrow, c8 & 7), b);
            mma_16816(o[2 * dq], pa, b[0], b[1]);
            mma_16816(o[2 * dq + 1], pa, b[2], b[3]);
          }
        }
      }
      cp_async_wait_all();
      if (kt + 1 < nkt && convert_cached(kt + 1)) __syncthreads();
      __syncthreads();  // tile kt+1 landed; every warp is done with tile kt's buffer
    }
    if (active) {
      l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
      l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
      l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
      l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
      float inv_a = 1.f / l_a, inv_b = 1.f / l_b;
      // a non-finite sum (a query or key value past the f16 range reached the
      // row) or a largest logit past kExactLogit: this lane's columns of the row
      // are recomputed in fp32
      for (int w = 0; w < 2; ++w) {
        const int rr = w ? rb : ra;
        if (rr < rows && !((w ? l_b : l_a) <= 3.0e38f && (w ? m_b : m_a) <= kExactLogit)) {
          float ex[D / 4];
          const int tt = w ? ttb : tta;
          if (!exact_row<D, D / 4>(prm.ex, p, t0 + tt, g * G + (rr - tt * G), w ? lo_b : lo_a,
                                   w ? lim_b : lim_a, 2 * (lane & 3), 8, ex))
            report(prm.status, GIST_ATTN_STATUS_RANGE);
#pragma unroll
          for (int dn = 0; dn < D / 8; ++dn) {
            o[dn][2 * w] = ex[2 * dn];
            o[dn][2 * w + 1] = ex[2 * dn + 1];
          }
          if (w) inv_b = 1.f; else inv_a = 1.f;
        }
      }
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        const uint32_t panel = sQ + (dn >> 3) * prm.q_panel + (lane & 3) * 4;
        sts32(panel + swz128(ra, dn & 7), float2_to_bf16x2(o[dn][0] * inv_a, o[dn][1] * inv_a));
        sts32(panel + swz128(rb, dn & 7), float2_to_bf16x2(o[dn][2] * inv_b, o[dn][3] * inv_b));
      }
    }
  } else {
    for (int idx = tid; idx < NP * prm.Tg * G * 8; idx += kThreads) {
      const int pn = idx / (prm.Tg * G * 8), r = idx % (prm.Tg * G * 8);
      sts16(sQ + pn * prm.q_panel + (uint32_t)r * 16, make_uint4(0, 0, 0, 0));
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {
    if (bad) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
#pragma unroll
    for (int pn = 0; pn < NP; ++pn) tma_store_5d(&tm_o, sQ + pn * prm.q_panel, 0, pn, g * G, t0, p);
    bulk_commit();
    bulk_wait_read_all();
  }
}

int encode_map(CUtensorMap* m, const void* base, const Problem& pb, int T) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return GIST_ATTN_ERR_LAUNCH;
  const cuuint64_t dims[5] = {64, (cuuint64_t)(pb.d / 64), (cuuint64_t)pb.Hq, (cuuint64_t)pb.l,
                              (cuuint64_t)pb.P};
  const cuuint64_t strides[4] = {128, (cuuint64_t)pb.d * 2, (cuuint64_t)pb.Hq * pb.d * 2,
                                 (cuuint64_t)pb.l * pb.Hq * pb.d * 2};
  const cuuint32_t box[5] = {64, 1, (cuuint32_t)pb.G, (cuuint32_t)T, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GIST_ATTN_OK : GIST_ATTN_ERR_UNSUPPORTED;
}

template <int D>
int launch_d(const Problem& pb, cudaStream_t stream) {
  const Layout L = plan(pb);
  if (L.bytes > (uint32_t)kMaxSmem) return GIST_ATTN_ERR_UNSUPPORTED;
  StreamParams prm{};
  prm.k_new = static_cast<const bf16*>(pb.k_new);
  prm.v_new = static_cast<const bf16*>(pb.v_new);
  prm.pv = PoolView{static_cast<const bf16*>(pb.kv_pool), pb.item_ids, pb.block_table,
                    pb.blocks_per_pair, pb.block_len, pb.num_blocks, pb.L, pb.layer, pb.Hkv, pb.d};
  prm.pos_offset = pb.pos_offset;
  prm.gist_start = pb.gist_start;
  prm.gist_len = pb.gist_len;
  prm.status = pb.status;
  prm.l = pb.l;
  prm.Hkv = pb.Hkv;
  prm.G = pb.G;
  prm.C = pb.C;
  prm.Tg = L.Tg;
  prm.ngroups = L.ngroups;
  prm.off_ring = L.off_ring;
  prm.ring_buf = L.ring_buf;
  prm.off_rt = L.off_rt;
  prm.off_bq = L.off_bq;
  prm.off_bk = L.off_bk;
  prm.off_ids = L.off_ids;
  prm.off_bar = L.off_bar;
  prm.q_panel = L.q_panel;
  prm.scale_log2 = pb.scale_log2;
  for (int j = 0; j < 64; ++j) prm.inv_freq[j] = pb.inv_freq[j];
  exact_inputs_from(prm.ex, pb);
  alignas(64) CUtensorMap tm_q, tm_o;
  int rc = encode_map(&tm_q, pb.q, pb, L.Tg);
  if (rc != GIST_ATTN_OK) return rc;
  rc = encode_map(&tm_o, pb.out, pb, L.Tg);
  if (rc != GIST_ATTN_OK) return rc;
  if (cudaFuncSetAttribute(prefill_stream_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)L.bytes) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  const int64_t grid = (int64_t)pb.P * pb.Hkv * L.ngroups;
  if (grid > 0x7fffffff) return GIST_ATTN_ERR_UNSUPPORTED;
  prefill_stream_kernel<D><<<(unsigned)grid, kThreads, L.bytes, stream>>>(tm_q, tm_o, prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

}  // namespace

// Any cache length and any l; groups of at most 64 query heads per KV head.
bool prefill_fits(const Problem& pb) {
  return pb.G <= kRowsMax && pb.blocks_per_pair <= 4096 && plan(pb).bytes <= (uint32_t)kMaxSmem;
}

int launch_prefill(const Problem& pb, cudaStream_t stream) {
  if (pb.d == 64) return launch_d<64>(pb, stream);
  if (pb.d == 128) return launch_d<128>(pb, stream);
  return GIST_ATTN_ERR_UNSUPPORTED;
}

}  // namespace gattn
