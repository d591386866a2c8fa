// gemm.cu -- the projections on either side of the attention, on the
// 5th-generation tensor core: the QKV projection with RoPE in its epilogue,
// and the output projection.
//
// [Gist page, "在线的一次 attention"]: per layer the new tokens' hidden states
// are projected to Q, K, V, the attention runs against the cached segment, and
// its output goes through the output projection.  Both projections are
// C[M][N] = A[M][K] B[N][K]^T with bf16 inputs and fp32 accumulation.  In the
// QKV epilogue the query and key heads are rotated at their positions from the
// fp32 accumulator (rotate-half RoPE) before the one rounding to bf16, so the
// attention can take them as they are.
//
// Persistent CTAs, one per SM, warp-specialised: warp 4 streams 128 x 64
// tiles of A and 256 x 64 tiles of B by TMA (128-byte swizzle) through a
// 4-stage ring (3 where the RoPE table leaves no room for a fourth), warp 5
// issues tcgen05.mma (128 x 256 x 16) into one of two 256-column TMEM
// accumulators, and warps 0-3 (one thread per output row) drain the other:
// RoPE, bf16, then one 32-row x 64-column box per warp in shared memory, stored
// by TMA while the next box is computed.  Output tiles run along N first, so
// the 128-row strip of A a CTA reads stays in L2.
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上".
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace gattn {
namespace {

constexpr int kEpi = 128;            // epilogue threads: one per tile row
constexpr int kThreads = kEpi + 64;  // + the TMA warp and the MMA warp
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr uint32_t kTileA = kBM * kBK * 2;    // bytes of one A k-block tile
constexpr uint32_t kTileB = kBN * kBK * 2;    // bytes of one B k-block tile
constexpr uint32_t kStage = kTileA + kTileB;
constexpr uint32_t kSlot = 32 * 128;          // one warp's 32 rows x 64 columns of bf16
constexpr int kMaxSlots = 8;                  // pairs one 128-row tile can touch (QKV mode)
constexpr int kMaxStages = 4;
constexpr int kMaxSmem = 227 * 1024;

// 2-D tiled store from shared memory (elements outside the tensor are dropped).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}

// After tcgen05.wait::ld: makes every use of the loaded registers depend on
// the wait, so several TMEM loads can be in flight before one wait.
__device__ __forceinline__ void tmem_pin(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                 "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

struct GemmParams {
  int M, N, K;
  int qkv;  // 0: y[M][N]; 1: split into q / k_new / v_new, rotating q and k
  int l, Hq, Hkv, C;
  const int32_t* pos_offset;
  int32_t* status;
  int ntn, num_tiles;
  int slots;     // pairs one 128-row tile can touch: (127 / l) + 2, at most kMaxSlots
  int tab_rows;  // 8 + ceil(l / 8): the two levels of the token-angle table
  uint32_t off_out, off_tab, tab_stride, off_base, off_bar;
  double theta[64];  // RoPE frequencies (angles reduced in double)
};

struct GBars {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_slot;
};

// tm_o0 / tm_o1 / tm_o2: q / k_new / v_new (QKV mode) or y (tm_o0 only), each
// [rows][columns] bf16 with 64 x 32 boxes.
// S: stages of the operand ring (4 where shared memory allows, else 3).
template <int D, int S>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_o0, const __grid_constant__ CUtensorMap tm_o1,
                const __grid_constant__ CUtensorMap tm_o2, const __grid_constant__ GemmParams prm) {
  constexpr int HALF = D / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  GBars* bars = reinterpret_cast<GBars*>(smem + prm.off_bar);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KB = (prm.K + kBK - 1) / kBK;
  const int my_tiles = (int)blockIdx.x < prm.num_tiles
                           ? (prm.num_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1
                           : 0;

  if (warp == 5) {
    tc::tmem_alloc(smem_u32(&bars->tmem_slot), 2 * kBN);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->acc_full[b], 1);
      mbar_init(&bars->acc_empty[b], kEpi);
    }
    fence_mbar_init();
  }
  if (prm.qkv) {
    // (cos, cos, sin, sin) of t theta for frequency pairs, in two levels: rows
    // 0..7 hold t = b < 8, rows 8.. hold t = 8a (a token's angle is the sum)
    for (int idx = tid; idx < prm.tab_rows * (HALF / 2); idx += kThreads) {
      const int row = idx / (HALF / 2), jp = idx - row * (HALF / 2);
      const int t = row < 8 ? row : 8 * (row - 8);
      float s0, c0, s1, c1;
      sincosf(rope_reduce(t, prm.theta[2 * jp]), &s0, &c0);
      sincosf(rope_reduce(t, prm.theta[2 * jp + 1]), &s1, &c1);
      *reinterpret_cast<float4*>(smem + prm.off_tab + row * prm.tab_stride + jp * 16) =
          make_float4(c0, c1, s0, s1);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_slot;

  if (warp == 4) {
    // ================================================================ TMA
    bool failed = false;
    if (lane == 0) {
      tma_prefetch_map(&tm_a);
      tma_prefetch_map(&tm_b);
    }
    int it = 0;  // k-blocks issued so far: ring slot it % S
    for (int tl = 0; tl < my_tiles && !failed; ++tl) {
      const int tile = (int)blockIdx.x + tl * (int)gridDim.x;
      const int m0 = (tile / prm.ntn) * kBM, n0 = (tile % prm.ntn) * kBN;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % S;
        // the slot is free once the MMAs that read it are done (a fresh
        // barrier passes the first wait)
        if (__any_sync(0xffffffffu,
                       !mbar_wait(&bars->empty[s], ((uint32_t)(it / S) & 1u) ^ 1u))) {
          failed = true;
          break;
        }
        if (lane == 0) {
          // rows of B past N (a narrower last tile) are zero-filled and counted
          mbar_arrive_expect_tx(&bars->full[s], kStage);
          tma_load_2d(sbase + s * kStage, &tm_a, &bars->full[s], kb * kBK, m0);
          tma_load_2d(sbase + s * kStage + kTileA, &tm_b, &bars->full[s], kb * kBK, n0);
        }
        __syncwarp();
      }
    }
    if (lane == 0 && failed) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
  } else if (warp == 5) {
    // ================================================================ MMA
    bool failed = false;
    int it = 0;
    for (int tl = 0; tl < my_tiles && !failed; ++tl) {
      const int b = tl & 1;
      const int tile = (int)blockIdx.x + tl * (int)gridDim.x;
      const int width = min(kBN, prm.N - (tile % prm.ntn) * kBN);
      const uint32_t idesc = tc::idesc_bf16_f32(kBM, (uint32_t)width, 0);
      if (__any_sync(0xffffffffu,
                     !mbar_wait(&bars->acc_empty[b], ((uint32_t)(tl >> 1) & 1u) ^ 1u))) {
        failed = true;
        break;
      }
      tc::fence_after_sync();
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % S;
        if (__any_sync(0xffffffffu, !mbar_wait(&bars->full[s], (uint32_t)(it / S) & 1u))) {
          failed = true;
          break;
        }
        tc::fence_after_sync();
        if (lane == 0) {
          const uint32_t a0 = sbase + s * kStage, b0 = a0 + kTileA;
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks) {
            const uint64_t ad = tc::smem_desc_sw128(a0 + ks * 32, 16, 1024);
            const uint64_t bd = tc::smem_desc_sw128(b0 + ks * 32, 16, 1024);
            tc::mma_ss(tmem + b * kBN, ad, bd, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
          }
          tc::commit(smem_u32(&bars->empty[s]));
          if (kb == KB - 1) tc::commit(smem_u32(&bars->acc_full[b]));
        }
        __syncwarp();
      }
    }
    if (lane == 0 && failed) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
  } else {
    // ================================================================ epilogue
    const int r = tid;  // tile row == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t out = sbase + prm.off_out + warp * kSlot;  // this warp's 32 x 64 output box
    const uint8_t* tab = smem + prm.off_tab;
    uint8_t* base = smem + prm.off_base;  // [slots][HALF / 2] of (cos, cos, sin, sin)
    const int rot_end = prm.qkv ? (prm.Hq + prm.Hkv) * D : 0;  // columns before it are rotated
    bool failed = false;
    if (lane == 0) {
      tma_prefetch_map(&tm_o0);
      if (prm.qkv) {
        tma_prefetch_map(&tm_o1);
        tma_prefetch_map(&tm_o2);
      }
    }
    for (int tl = 0; tl < my_tiles; ++tl) {
      const int b = tl & 1;
      const int tile = (int)blockIdx.x + tl * (int)gridDim.x;
      const int m0 = (tile / prm.ntn) * kBM, n0 = (tile % prm.ntn) * kBN;
      const int width = min(kBN, prm.N - n0);
      // the first position of each pair the tile touches (uniform branch)
      const uint8_t* tlo = tab;  // angle of t mod 8
      const uint8_t* thi = tab;  // angle of 8 (t / 8)
      const uint8_t* brow = base;
      if (n0 < rot_end) {
        const int p_first = m0 / prm.l;
        named_bar_sync(1, kEpi);  // every thread is done with the previous tile's slots
        for (int idx = r; idx < prm.slots * (HALF / 2); idx += kEpi) {
          const int sl = idx / (HALF / 2), jp = idx - sl * (HALF / 2);
          const int p = p_first + sl;
          if (p * prm.l < prm.M) {
            const int pos = prm.pos_offset ? prm.pos_offset[p] : prm.C;
            float s0, c0, s1, c1;
            sincosf(rope_reduce(pos, prm.theta[2 * jp]), &s0, &c0);
            sincosf(rope_reduce(pos, prm.theta[2 * jp + 1]), &s1, &c1);
            *reinterpret_cast<float4*>(base + idx * 16) = make_float4(c0, c1, s0, s1);
          }
        }
        named_bar_sync(1, kEpi);
        const int m = m0 + r;
        const int p = m / prm.l;
        const int t = m - p * prm.l;
        tlo = tab + (t & 7) * prm.tab_stride;
        thi = tab + (8 + (t >> 3)) * prm.tab_stride;
        brow = base + (p - p_first) * (HALF / 2) * 16;
      }
      if (!failed && !mbar_wait(&bars->acc_full[b], (uint32_t)(tl >> 1) & 1u)) failed = true;
      tc::fence_after_sync();
      const uint32_t acc = tmem + lane_base + b * kBN;
      // x' = x cos - y sin or y' = y cos + x sin for 16 columns, frequencies j0..j0+15
      auto rotate16 = [&](const uint32_t (&xv)[16], const uint32_t (&yv)[16], int j0, bool second,
                          uint32_t (&w)[8]) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int jp = (j0 >> 1) + e;
          const uint4 ls = *reinterpret_cast<const uint4*>(tlo + jp * 16);
          const uint4 hs = *reinterpret_cast<const uint4*>(thi + jp * 16);
          const uint4 bs = *reinterpret_cast<const uint4*>(brow + jp * 16);
          const uint64_t lc2 = f2_make(__uint_as_float(ls.x), __uint_as_float(ls.y));
          const uint64_t ls2 = f2_make(__uint_as_float(ls.z), __uint_as_float(ls.w));
          const uint64_t hc2 = f2_make(__uint_as_float(hs.x), __uint_as_float(hs.y));
          const uint64_t hs2 = f2_make(__uint_as_float(hs.z), __uint_as_float(hs.w));
          // angle of t = angle(8 (t / 8)) + angle(t mod 8)
          const uint64_t tc2 = f2_sub(f2_mul(hc2, lc2), f2_mul(hs2, ls2));
          const uint64_t ts2 = f2_fma(hs2, lc2, f2_mul(hc2, ls2));
          const uint64_t bc2 = f2_make(__uint_as_float(bs.x), __uint_as_float(bs.y));
          const uint64_t bs2 = f2_make(__uint_as_float(bs.z), __uint_as_float(bs.w));
          // angle of position pos0 + t = angle(pos0) + angle(t)
          const uint64_t cc = f2_sub(f2_mul(bc2, tc2), f2_mul(bs2, ts2));
          const uint64_t ss = f2_fma(bs2, tc2, f2_mul(bc2, ts2));
          const uint64_t x = f2_make(__uint_as_float(xv[2 * e]), __uint_as_float(xv[2 * e + 1]));
          const uint64_t y = f2_make(__uint_as_float(yv[2 * e]), __uint_as_float(yv[2 * e + 1]));
          w[e] = second ? f2_to_bf16x2(f2_fma(y, cc, f2_mul(x, ss)))
                        : f2_to_bf16x2(f2_sub(f2_mul(x, cc), f2_mul(y, ss)));
        }
      };
      // one 64-column box at a time: computed, written to the warp's box once the
      // previous box's store has read it, and stored by TMA
      for (int j = 0; j < width / 64; ++j) {
        const int nb = n0 + 64 * j;  // first column of the box
        const CUtensorMap* map = &tm_o0;
        int col = nb;
        if (prm.qkv && nb >= prm.Hq * D) {
          if (nb < rot_end) {
            map = &tm_o1;
            col = nb - prm.Hq * D;
          } else {
            map = &tm_o2;
            col = nb - rot_end;
          }
        }
        const uint32_t a0 = acc + 64 * j;
        uint32_t w[4][8];
        if (nb >= rot_end) {
          uint32_t v[4][16];
#pragma unroll
          for (int q = 0; q < 4; ++q) tc::ld16(a0 + 16 * q, v[q]);
          tc::wait_ld();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            tmem_pin(v[q]);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[q][e] = f2_to_bf16x2(f2_make(__uint_as_float(v[q][2 * e]), __uint_as_float(v[q][2 * e + 1])));
          }
        } else if (D == 64) {
          // the box is one head: x = columns 0..31, y = 32..63
          uint32_t v[4][16];
#pragma unroll
          for (int q = 0; q < 4; ++q) tc::ld16(a0 + 16 * q, v[q]);
          tc::wait_ld();
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_pin(v[q]);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            rotate16(v[q], v[q + 2], 16 * q, false, w[q]);
            rotate16(v[q], v[q + 2], 16 * q, true, w[q + 2]);
          }
        } else {
          // half of a 128-column head: x' from the first box (j even), y' from the second
          const bool second = (j & 1) != 0;
          const uint32_t hx = second ? a0 - 64 : a0;  // the head's x columns
#pragma unroll
          for (int q2 = 0; q2 < 4; q2 += 2) {
            uint32_t xv[2][16], yv[2][16];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              tc::ld16(hx + 16 * (q2 + q), xv[q]);
              tc::ld16(hx + 64 + 16 * (q2 + q), yv[q]);
            }
            tc::wait_ld();
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              tmem_pin(xv[q]);
              tmem_pin(yv[q]);
              rotate16(xv[q], yv[q], 16 * (q2 + q), second, w[q2 + q]);
            }
          }
        }
        if (lane == 0) bulk_wait_read_all();  // the previous box has been read out
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          sts16(out + swz128(lane, 2 * q), make_uint4(w[q][0], w[q][1], w[q][2], w[q][3]));
          sts16(out + swz128(lane, 2 * q + 1), make_uint4(w[q][4], w[q][5], w[q][6], w[q][7]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {  // rows past M are dropped by the store
          tma_store_2d(map, out, col, m0 + warp * 32);
          bulk_commit();
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&bars->acc_empty[b]);
    }
    if (lane == 0) bulk_wait_all();
    if (failed && r == 0) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 2 * kBN);
  }
}

// Row-major [rows][cols] bf16, boxes of box_cols x box_rows, 128-byte swizzle.
int encode_2d(CUtensorMap* m, const void* base, int64_t rows, int cols, int box_cols, int box_rows) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return GIST_ATTN_ERR_LAUNCH;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GIST_ATTN_OK : GIST_ATTN_ERR_UNSUPPORTED;
}

// Shared memory: the ring of S stages, the output boxes, the RoPE table of l rows
// and the per-tile base slots; 0 if it does not fit.
uint32_t smem_plan(GemmParams& prm, int d, int stages) {
  uint32_t off = (uint32_t)stages * kStage;
  prm.off_out = off;
  off += 4 * kSlot;
  prm.off_tab = off;
  prm.tab_stride = (uint32_t)(d / 4) * 16 + 16;  // +16 B: consecutive tokens on different banks
  off += prm.qkv ? (uint32_t)prm.tab_rows * prm.tab_stride : 0;
  prm.off_base = off;
  off += prm.qkv ? (uint32_t)prm.slots * (d / 4) * 16 : 0;
  prm.off_bar = off;
  off += 128;
  const uint32_t bytes = off + 1024;
  return bytes <= (uint32_t)kMaxSmem ? bytes : 0;
}

template <int D, int S>
int launch_gemm_d(GemmParams prm, const void* a, const void* b, void* o0, void* o1, void* o2,
                  cudaStream_t stream) {
  const uint32_t bytes = smem_plan(prm, D, S);
  if (bytes == 0) return GIST_ATTN_ERR_UNSUPPORTED;
  alignas(64) CUtensorMap tm_a, tm_b, tm_o0, tm_o1, tm_o2;
  int rc = encode_2d(&tm_a, a, prm.M, prm.K, kBK, kBM);
  if (rc == GIST_ATTN_OK) rc = encode_2d(&tm_b, b, prm.N, prm.K, kBK, kBN);
  if (prm.qkv) {
    if (rc == GIST_ATTN_OK) rc = encode_2d(&tm_o0, o0, prm.M, prm.Hq * D, 64, 32);
    if (rc == GIST_ATTN_OK) rc = encode_2d(&tm_o1, o1, prm.M, prm.Hkv * D, 64, 32);
    if (rc == GIST_ATTN_OK) rc = encode_2d(&tm_o2, o2, prm.M, prm.Hkv * D, 64, 32);
  } else {
    if (rc == GIST_ATTN_OK) rc = encode_2d(&tm_o0, o0, prm.M, prm.N, 64, 32);
    tm_o1 = tm_o0;
    tm_o2 = tm_o0;
  }
  if (rc != GIST_ATTN_OK) return rc;
  if (cudaFuncSetAttribute(gemm_kernel<D, S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  const int grid = prm.num_tiles < sms ? prm.num_tiles : sms;
  gemm_kernel<D, S><<<grid, kThreads, bytes, stream>>>(tm_a, tm_b, tm_o0, tm_o1, tm_o2, prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

// Four stages where they fit beside the output boxes and the RoPE table, else three.
template <int D>
int launch_gemm_stages(GemmParams prm, const void* a, const void* b, void* o0, void* o1,
                       void* o2, cudaStream_t stream) {
  GemmParams probe = prm;
  if (smem_plan(probe, D, 4) != 0) return launch_gemm_d<D, 4>(prm, a, b, o0, o1, o2, stream);
  return launch_gemm_d<D, 3>(prm, a, b, o0, o1, o2, stream);
}

int launch_common(GemmParams& prm, const void* a, const void* b, int d, void* o0, void* o1,
                  void* o2, cudaStream_t stream) {
  const int64_t mt = ((int64_t)prm.M + kBM - 1) / kBM;
  prm.ntn = (prm.N + kBN - 1) / kBN;
  if (mt * prm.ntn > 0x7fffffff) return GIST_ATTN_ERR_UNSUPPORTED;
  prm.num_tiles = (int)(mt * prm.ntn);
  if (prm.num_tiles == 0) return GIST_ATTN_OK;
  if (d == 64) return launch_gemm_stages<64>(prm, a, b, o0, o1, o2, stream);
  return launch_gemm_stages<128>(prm, a, b, o0, o1, o2, stream);
}

}  // namespace

// Sizes this build runs: N a multiple of 128 (whole 128-column units), K a
// multiple of 8 (16-byte rows for TMA), M below 2^31; for the QKV split also
// q and k/v sections made of whole units.
bool gemm_fits(int64_t M, int N, int K) {
  return M >= 0 && M < 0x7fffffff && N > 0 && N % 128 == 0 && K > 0 && K % 8 == 0;
}

int launch_qkv_rope(const Problem& pb, const void* x, const void* w, int d_model, void* q,
                    void* kn, void* vn, cudaStream_t stream) {
  GemmParams prm{};
  prm.M = pb.P * pb.l;
  prm.N = (pb.Hq + 2 * pb.Hkv) * pb.d;
  prm.K = d_model;
  if (!gemm_fits((int64_t)pb.P * pb.l, prm.N, prm.K)) return GIST_ATTN_ERR_UNSUPPORTED;
  // every 128-column unit must lie inside one of the q / k / v sections
  if ((pb.Hq * pb.d) % 128 != 0 || (pb.Hkv * pb.d) % 128 != 0) return GIST_ATTN_ERR_UNSUPPORTED;
  // a 128-row tile must touch at most kMaxSlots pairs (the table's size is checked with
  // the shared-memory plan)
  if ((kBM - 1) / pb.l + 2 > kMaxSlots) return GIST_ATTN_ERR_UNSUPPORTED;
  prm.qkv = 1;
  prm.slots = (kBM - 1) / pb.l + 2;
  prm.tab_rows = 8 + (pb.l + 7) / 8;
  prm.l = pb.l;
  prm.Hq = pb.Hq;
  prm.Hkv = pb.Hkv;
  prm.C = pb.C;
  prm.pos_offset = pb.pos_offset;
  prm.status = pb.status;
  for (int j = 0; j < 64; ++j) prm.theta[j] = pb.inv_freq_d[j];
  return launch_common(prm, x, w, pb.d, q, kn, vn, stream);
}

int launch_out_proj(const Problem& pb, const void* attn, const void* w, int d_model, void* y,
                    cudaStream_t stream) {
  GemmParams prm{};
  prm.M = pb.P * pb.l;
  prm.N = d_model;
  prm.K = pb.Hq * pb.d;
  if (!gemm_fits((int64_t)pb.P * pb.l, prm.N, prm.K)) return GIST_ATTN_ERR_UNSUPPORTED;
  prm.qkv = 0;
  prm.status = pb.status;
  prm.l = pb.l;
  return launch_common(prm, attn, w, 64, y, nullptr, nullptr, stream);
}

}  // namespace gattn
