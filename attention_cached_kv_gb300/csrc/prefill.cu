// prefill.cu -- attention of l >= 2 new tokens against a pair's cached
// segment, one CTA per (pair, KV head, chunk of new tokens).
//
// [Gist page, "在线的一次 attention"]: K = cat(cache[item].K[layer], K_new),
// V likewise; the query is numbered after the k cached positions; causal
// inside the new block; nothing is written back.  [Gist page, "收益有多大：存储"]:
// K/V are stored per KV head and shared by that head's group of Hq/Hkv query
// heads, so one CTA serves the whole group: its rows are (token, head-in-group)
// pairs, token-major, which is exactly how q/out are laid out in memory
// ([P][l][Hq][d], the group's heads adjacent).  [Gist page, "收益有多大：算力"]:
// only the K.Q logits, the softmax and softmax x V depend on the KV length;
// those three are this kernel.
//
// Data movement (per CTA):
//   Q   [T tokens][G heads][d] -> shared memory by one TMA tensor copy per
//       64-column panel, 128-byte swizzle (conflict-free ldmatrix);
//   K/V cached rows            -> 16-byte cp.async through the pool gather;
//   V_new rows                 -> 16-byte cp.async;
//   K_new rows                 -> registers, RoPE at their positions, st.shared;
//   O                          -> written over the Q rows the warp consumed,
//                                 then one TMA tensor store per panel.
// Compute: each warp takes 16-row tiles; Q fragments are rotated in
// registers, S = Q K^T and O += P V run on mma.sync m16n8k16 (bf16 in, fp32
// accumulate) over 64-key blocks with an online (running max / sum) softmax.
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上".
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace gattn {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kQBudgetBytes = 64 * 1024;  // Q/O tile per CTA
constexpr int kMaxSmem = 227 * 1024;

struct PrefillParams {
  const bf16* k_new;
  const bf16* v_new;
  PoolView pv;
  const int32_t* pos_offset;
  int32_t* status;
  int P, l, Hkv, G, C;
  int T, n_chunks;
  int q_rows_alloc;   // rows per Q/O panel (multiple of 16)
  int kv_rows_alloc;  // rows per K (and V) panel (multiple of 16)
  uint32_t off_k, off_v, off_tab, off_ids, off_bar;
  float scale_log2;
  float inv_freq[64];
};

struct Layout {
  int T, n_chunks, q_rows_alloc, kv_rows_alloc;
  uint32_t off_k, off_v, off_tab, off_ids, off_bar, bytes;
};

Layout plan(const Problem& pb) {
  Layout L{};
  const int row_bytes = pb.G * pb.d * 2;  // one token of the head group
  int tmax = kQBudgetBytes / row_bytes;
  if (tmax < 1) tmax = 1;
  if (tmax > 256) tmax = 256;
  L.n_chunks = (pb.l + tmax - 1) / tmax;
  L.T = (pb.l + L.n_chunks - 1) / L.n_chunks;  // balanced chunks
  const int np = pb.d / 64;
  L.q_rows_alloc = (L.T * pb.G + 15) / 16 * 16;
  L.kv_rows_alloc = (pb.C + pb.l + 15) / 16 * 16;
  uint32_t off = (uint32_t)np * L.q_rows_alloc * 128;
  L.off_k = off;
  off += (uint32_t)np * L.kv_rows_alloc * 128;
  L.off_v = off;
  off += (uint32_t)np * L.kv_rows_alloc * 128;
  L.off_tab = off;
  off += (uint32_t)L.T * (pb.d / 2) * 8;
  L.off_ids = off;
  off += ((uint32_t)pb.blocks_per_pair * 4 + 15) / 16 * 16;
  L.off_bar = off;
  off += 16;
  L.bytes = off + 1024;  // slack to align the base to 1024 bytes
  return L;
}

template <int D>
__global__ void __launch_bounds__(kThreads)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                   const __grid_constant__ PrefillParams prm) {
  constexpr int NP = D / 64;    // 128-byte panels per row
  constexpr int CPR = D / 8;    // 16-byte chunks per row
  constexpr int HALF = D / 2;
  constexpr float kNegInf = -INFINITY;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + prm.off_k;
  const uint32_t sV = sQ + prm.off_v;
  float2* tab = reinterpret_cast<float2*>(smem + prm.off_tab);
  int32_t* ids = reinterpret_cast<int32_t*>(smem + prm.off_ids);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + prm.off_bar);
  const uint32_t q_panel = (uint32_t)prm.q_rows_alloc * 128;
  const uint32_t kv_panel = (uint32_t)prm.kv_rows_alloc * 128;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int unit = blockIdx.x;
  const int chunk = unit % prm.n_chunks;
  unit /= prm.n_chunks;
  const int g = unit % prm.Hkv;
  const int p = unit / prm.Hkv;
  const int G = prm.G, C = prm.C, l = prm.l;
  const int t0 = chunk * prm.T;
  const int Tc = min(prm.T, l - t0);  // tokens of this chunk
  const int rows = Tc * G;
  const int nnew = t0 + Tc;           // new keys any row here may see
  const int nk = C + nnew;
  const int nk16 = (nk + 15) & ~15;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_o);
    mbar_arrive_expect_tx(bar, (uint32_t)NP * prm.T * G * 128);
#pragma unroll
    for (int pn = 0; pn < NP; ++pn) tma_load_5d(sQ + pn * q_panel, &tm_q, bar, 0, pn, g * G, t0, p);
  }

  // Block ids of this pair, checked once.
  bool bad = false;
  for (int b = tid; b < prm.pv.blocks_per_pair; b += kThreads) {
    const int32_t blk = pool_block_id(prm.pv, p, b);
    bad |= !pool_block_ok(prm.pv, blk);
    ids[b] = blk;
  }
  // cos/sin of this chunk's positions: tab[tt][j] = (cos, sin)(pos(t0 + tt) * theta_j)
  const int pos_base = prm.pos_offset ? prm.pos_offset[p] : C;  // position of new token 0
  for (int idx = tid; idx < Tc * HALF; idx += kThreads) {
    const int tt = idx / HALF, j = idx - tt * HALF;
    float s, c;
    sincosf((float)(pos_base + t0 + tt) * prm.inv_freq[j], &s, &c);
    tab[idx] = make_float2(c, s);
  }
  bad = __syncthreads_or(bad);

  if (!bad) {
    const int bl = prm.pv.block_len;
    // cached K and V rows
    const int cached_chunks = C * CPR;
    for (int idx = tid; idx < 2 * cached_chunks; idx += kThreads) {
      const int kv = idx >= cached_chunks;
      const int r = idx - kv * cached_chunks;
      const int kappa = r / CPR, c = r - kappa * CPR;
      const int b = kappa / bl, t = kappa - b * bl;
      const bf16* src = pool_row(prm.pv, ids[b], g, kv, t) + c * 8;
      cp_async16((kv ? sV : sK) + (c >> 3) * kv_panel + swz128(kappa, c & 7), src);
    }
    // new V rows 0 .. nnew-1 at keys C ..
    for (int idx = tid; idx < nnew * CPR; idx += kThreads) {
      const int t = idx / CPR, c = idx - t * CPR;
      const bf16* src = prm.v_new + (((int64_t)p * l + t) * prm.Hkv + g) * D + c * 8;
      cp_async16(sV + (c >> 3) * kv_panel + swz128(C + t, c & 7), src);
    }
    cp_async_commit();
    // new K rows, rotated at their own positions (rotate-half pairs j, j + d/2)
    for (int idx = tid; idx < nnew * (CPR / 2); idx += kThreads) {
      const int t = idx / (CPR / 2), c = idx - t * (CPR / 2);
      const bf16* src = prm.k_new + (((int64_t)p * l + t) * prm.Hkv + g) * D;
      uint4 lo = ldg16(src + c * 8), hi = ldg16(src + HALF + c * 8);
      uint32_t* lw = reinterpret_cast<uint32_t*>(&lo);
      uint32_t* hw = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = c * 8 + 2 * e;
        float c0, s0, c1, s1;
        if (t >= t0) {
          const float2 a = tab[(t - t0) * HALF + j], b2 = tab[(t - t0) * HALF + j + 1];
          c0 = a.x; s0 = a.y; c1 = b2.x; s1 = b2.y;
        } else {
          sincosf((float)(pos_base + t) * prm.inv_freq[j], &s0, &c0);
          sincosf((float)(pos_base + t) * prm.inv_freq[j + 1], &s1, &c1);
        }
        const float2 x = bf16x2_to_float2(lw[e]), y = bf16x2_to_float2(hw[e]);
        lw[e] = float2_to_bf16x2(x.x * c0 - y.x * s0, x.y * c1 - y.y * s1);
        hw[e] = float2_to_bf16x2(y.x * c0 + x.x * s0, y.y * c1 + x.y * s1);
      }
      sts16(sK + (c >> 3) * kv_panel + swz128(C + t, c & 7), lo);
      const int ch = c + CPR / 2;
      sts16(sK + (ch >> 3) * kv_panel + swz128(C + t, ch & 7), hi);
    }
    // zero rows nk .. nk16-1 so padded keys contribute exactly nothing
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int idx = tid; idx < (nk16 - nk) * CPR * 2; idx += kThreads) {
      const int kv = idx >= (nk16 - nk) * CPR;
      const int r = idx - kv * (nk16 - nk) * CPR;
      const int row = nk + r / CPR, c = r % CPR;
      sts16((kv ? sV : sK) + (c >> 3) * kv_panel + swz128(row, c & 7), z);
    }
    cp_async_wait_all();
  }

  // Q tile landed?
  bool timed_out = !mbar_wait(bar, 0);
  timed_out = __syncthreads_or(timed_out);
  if (timed_out) {
    if (tid == 0) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
    mbar_wait(bar, 0);  // one more bounded wait for the copy in flight
    return;
  }

  if (bad) {
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int idx = tid; idx < NP * prm.T * G * 8; idx += kThreads) {
      const int pn = idx / (prm.T * G * 8), r = idx % (prm.T * G * 8);
      sts16(sQ + pn * q_panel + (uint32_t)r * 16, z);
    }
  } else {
    const float scale_log2 = prm.scale_log2;
    const int n_mt = (rows + 15) / 16;
    for (int mt = warp; mt < n_mt; mt += kWarps) {
      const int r0 = mt * 16;
      // ---- Q fragments (A operand, row-major 16 x d) + RoPE in registers
      uint32_t qa[D / 16][4];
      {
        const int row = r0 + (lane & 15);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int c8 = ks * 2 + (lane >> 4);
          ldsm_x4(sQ + (c8 >> 3) * q_panel + swz128(row, c8 & 7), qa[ks]);
        }
      }
      const int ra = r0 + (lane >> 2), rb = ra + 8;
      const int tta = min(ra / G, Tc - 1), ttb = min(rb / G, Tc - 1);
#pragma unroll
      for (int ks = 0; ks < D / 32; ++ks) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int tt = (r & 1) ? ttb : tta;
          const int j = ks * 16 + 2 * (lane & 3) + ((r & 2) ? 8 : 0);
          const float4 cs = *reinterpret_cast<const float4*>(&tab[tt * HALF + j]);
          const float2 x = bf16x2_to_float2(qa[ks][r]);
          const float2 y = bf16x2_to_float2(qa[ks + D / 32][r]);
          qa[ks][r] = float2_to_bf16x2(x.x * cs.x - y.x * cs.y, x.y * cs.z - y.y * cs.w);
          qa[ks + D / 32][r] = float2_to_bf16x2(y.x * cs.x + x.x * cs.y, y.y * cs.z + x.y * cs.w);
        }
      }
      // keys visible to rows ra / rb, and to the tile's last row
      const int lim_a = C + t0 + tta + 1, lim_b = C + t0 + ttb + 1;
      const int kmax = C + t0 + min((r0 + 15) / G, Tc - 1) + 1;

      float o[D / 8][4];
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
      float m_a = kNegInf, m_b = kNegInf, l_a = 0.f, l_b = 0.f;

      for (int kb = 0; kb < kmax; kb += 64) {
        const int nt = min(8, (kmax - kb + 7) >> 3);
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
          if (n < nt) {
            const int krow = kb + n * 8 + (lane & 7);
#pragma unroll
            for (int k2 = 0; k2 < D / 32; ++k2) {
              uint32_t b[4];
              const int c8 = k2 * 4 + (lane >> 3);
              ldsm_x4(sK + (c8 >> 3) * kv_panel + swz128(krow, c8 & 7), b);
              mma_16816(s[n], qa[2 * k2], b[0], b[1]);
              mma_16816(s[n], qa[2 * k2 + 1], b[2], b[3]);
            }
          }
        }
        // mask, scale (log2 units), running max
        float mx_a = kNegInf, mx_b = kNegInf;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int key = kb + n * 8 + 2 * (lane & 3);
          s[n][0] = key < lim_a ? s[n][0] * scale_log2 : kNegInf;
          s[n][1] = key + 1 < lim_a ? s[n][1] * scale_log2 : kNegInf;
          s[n][2] = key < lim_b ? s[n][2] * scale_log2 : kNegInf;
          s[n][3] = key + 1 < lim_b ? s[n][3] * scale_log2 : kNegInf;
          mx_a = fmaxf(mx_a, fmaxf(s[n][0], s[n][1]));
          mx_b = fmaxf(mx_b, fmaxf(s[n][2], s[n][3]));
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float al_a = exp2f(m_a - mn_a), al_b = exp2f(m_b - mn_b);
        m_a = mn_a;
        m_b = mn_b;
        float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          s[n][0] = exp2f(s[n][0] - mn_a);
          s[n][1] = exp2f(s[n][1] - mn_a);
          s[n][2] = exp2f(s[n][2] - mn_b);
          s[n][3] = exp2f(s[n][3] - mn_b);
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
        // O += P V, 16 keys per step
        const int nks = (nt + 1) >> 1;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if (kk < nks) {
            uint32_t pa[4];
            pa[0] = float2_to_bf16x2(s[2 * kk][0], s[2 * kk][1]);
            pa[1] = float2_to_bf16x2(s[2 * kk][2], s[2 * kk][3]);
            pa[2] = float2_to_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            pa[3] = float2_to_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            const int vrow = kb + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int dq = 0; dq < D / 16; ++dq) {
              uint32_t b[4];
              const int c8 = dq * 2 + (lane >> 4);
              ldsm_x4_trans(sV + (c8 >> 3) * kv_panel + swz128(vrow, c8 & 7), b);
              mma_16816(o[2 * dq], pa, b[0], b[1]);
              mma_16816(o[2 * dq + 1], pa, b[2], b[3]);
            }
          }
        }
      }
      // ---- normalise, round, write over this tile's Q rows
      l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
      l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
      l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
      l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
      const float inv_a = 1.f / l_a, inv_b = 1.f / l_b;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        const uint32_t panel = sQ + (dn >> 3) * q_panel + (lane & 3) * 4;
        sts32(panel + swz128(ra, dn & 7), float2_to_bf16x2(o[dn][0] * inv_a, o[dn][1] * inv_a));
        sts32(panel + swz128(rb, dn & 7), float2_to_bf16x2(o[dn][2] * inv_b, o[dn][3] * inv_b));
      }
    }
  }

  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {
    if (bad) report(prm.status, GIST_ATTN_STATUS_BAD_BLOCK);
#pragma unroll
    for (int pn = 0; pn < NP; ++pn) tma_store_5d(&tm_o, sQ + pn * q_panel, 0, pn, g * G, t0, p);
    bulk_commit();
    bulk_wait_read_all();
  }
}

// 5-D view [P][l][Hq][d/64][64] of q or out; box = one chunk of the head group.
int encode_qo_map(CUtensorMap* m, const void* base, const Problem& pb, int T) {
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
  PrefillParams prm{};
  prm.k_new = static_cast<const bf16*>(pb.k_new);
  prm.v_new = static_cast<const bf16*>(pb.v_new);
  prm.pv = PoolView{static_cast<const bf16*>(pb.kv_pool), pb.item_ids, pb.block_table,
                    pb.blocks_per_pair, pb.block_len, pb.num_blocks, pb.L, pb.layer, pb.Hkv, pb.d};
  prm.pos_offset = pb.pos_offset;
  prm.status = pb.status;
  prm.P = pb.P;
  prm.l = pb.l;
  prm.Hkv = pb.Hkv;
  prm.G = pb.G;
  prm.C = pb.C;
  prm.T = L.T;
  prm.n_chunks = L.n_chunks;
  prm.q_rows_alloc = L.q_rows_alloc;
  prm.kv_rows_alloc = L.kv_rows_alloc;
  prm.off_k = L.off_k;
  prm.off_v = L.off_v;
  prm.off_tab = L.off_tab;
  prm.off_ids = L.off_ids;
  prm.off_bar = L.off_bar;
  prm.scale_log2 = pb.scale_log2;
  for (int j = 0; j < 64; ++j) prm.inv_freq[j] = pb.inv_freq[j];

  alignas(64) CUtensorMap tm_q, tm_o;
  int rc = encode_qo_map(&tm_q, pb.q, pb, L.T);
  if (rc != GIST_ATTN_OK) return rc;
  rc = encode_qo_map(&tm_o, pb.out, pb, L.T);
  if (rc != GIST_ATTN_OK) return rc;

  if (cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)L.bytes) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  const int64_t grid = (int64_t)pb.P * pb.Hkv * L.n_chunks;
  if (grid > 0x7fffffff) return GIST_ATTN_ERR_UNSUPPORTED;
  prefill_kernel<D><<<(unsigned)grid, kThreads, L.bytes, stream>>>(tm_q, tm_o, prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

}  // namespace

bool prefill_fits(const Problem& pb) { return plan(pb).bytes <= (uint32_t)kMaxSmem; }

int launch_prefill(const Problem& pb, cudaStream_t stream) {
  if (pb.d == 64) return launch_d<64>(pb, stream);
  if (pb.d == 128) return launch_d<128>(pb, stream);
  return GIST_ATTN_ERR_UNSUPPORTED;
}

}  // namespace gattn
