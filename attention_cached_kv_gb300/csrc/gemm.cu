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
// Persistent CTAs, one per SM, warp-specialised: warp 4 streams 128 x 64 tiles
// of A and B by TMA (128-byte swizzle) through a 4-stage ring, warp 5 issues
// tcgen05.mma into one of two 128-column TMEM accumulators, and warps 0-3 (one
// thread per output row) drain the other accumulator: RoPE, bf16, 16-byte
// stores.  Output tiles run along N first, so the 128-row strip of A a CTA
// reads stays in L2 for the next tiles.
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
constexpr int kStages = 4;
constexpr int kBM = 128, kBN = 128, kBK = 64;
constexpr uint32_t kTile = kBM * kBK * 2;  // bytes of one A (or B) k-block tile
constexpr int kMaxSlots = 8;               // pairs one 128-row tile can touch (QKV mode)
constexpr int kMaxSmem = 227 * 1024;

struct GemmParams {
  int M, N, K;
  int qkv;        // 0: y[M][N]; 1: split into q / k_new / v_new, rotating q and k
  bf16* y;
  bf16* q;
  bf16* kn;
  bf16* vn;
  int l, Hq, Hkv, d, C;
  const int32_t* pos_offset;
  int32_t* status;
  int ntn, num_tiles;
  uint32_t off_tab, off_base, off_bar;
  float inv_freq[64];
};

struct GBars {
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_slot;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ GemmParams prm) {
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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->acc_full[b], 1);
      mbar_init(&bars->acc_empty[b], kEpi);
    }
    fence_mbar_init();
  }
  if (prm.qkv) {  // (cos, cos, sin, sin) of t theta for frequency pairs, t < l
    for (int idx = tid; idx < prm.l * (HALF / 2); idx += kThreads) {
      const int t = idx / (HALF / 2), jp = idx - t * (HALF / 2);
      float s0, c0, s1, c1;
      sincosf((float)t * prm.inv_freq[2 * jp], &s0, &c0);
      sincosf((float)t * prm.inv_freq[2 * jp + 1], &s1, &c1);
      *reinterpret_cast<float4*>(smem + prm.off_tab + (t * (HALF / 2) + jp) * 16) =
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
    int it = 0;  // k-blocks issued so far: ring slot it % kStages
    for (int tl = 0; tl < my_tiles && !failed; ++tl) {
      const int tile = (int)blockIdx.x + tl * (int)gridDim.x;
      const int m0 = (tile / prm.ntn) * kBM, n0 = (tile % prm.ntn) * kBN;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % kStages;
        // the slot is free once the MMAs that read it are done (a fresh
        // barrier passes the first wait)
        if (__any_sync(0xffffffffu,
                       !mbar_wait(&bars->empty[s], ((uint32_t)(it / kStages) & 1u) ^ 1u))) {
          failed = true;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->full[s], 2 * kTile);
          tma_load_2d(sbase + s * 2 * kTile, &tm_a, &bars->full[s], kb * kBK, m0);
          tma_load_2d(sbase + s * 2 * kTile + kTile, &tm_b, &bars->full[s], kb * kBK, n0);
        }
        __syncwarp();
      }
    }
    if (lane == 0 && failed) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
  } else if (warp == 5) {
    // ================================================================ MMA
    bool failed = false;
    int it = 0;
    const uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN, 0);
    for (int tl = 0; tl < my_tiles && !failed; ++tl) {
      const int b = tl & 1;
      if (__any_sync(0xffffffffu,
                     !mbar_wait(&bars->acc_empty[b], ((uint32_t)(tl >> 1) & 1u) ^ 1u))) {
        failed = true;
        break;
      }
      tc::fence_after_sync();
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % kStages;
        if (__any_sync(0xffffffffu, !mbar_wait(&bars->full[s], (uint32_t)(it / kStages) & 1u))) {
          failed = true;
          break;
        }
        tc::fence_after_sync();
        if (lane == 0) {
          const uint32_t a0 = sbase + s * 2 * kTile, b0 = a0 + kTile;
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
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint8_t* tab = smem + prm.off_tab;
    uint8_t* base = smem + prm.off_base;  // [kMaxSlots][HALF / 2] of (cos, cos, sin, sin)
    bool failed = false;
    for (int tl = 0; tl < my_tiles; ++tl) {
      const int b = tl & 1;
      const int tile = (int)blockIdx.x + tl * (int)gridDim.x;
      const int m0 = (tile / prm.ntn) * kBM, n0 = (tile % prm.ntn) * kBN;
      const int m = m0 + r;
      // what the tile's columns are: y, or q / k heads (rotated) / v heads
      int sect = 0;  // 0: y or v, 1: q or k (rotated)
      bf16* dst = nullptr;
      if (!prm.qkv) {
        dst = prm.y + (size_t)m * prm.N + n0;
      } else if (n0 < prm.Hq * D) {
        sect = 1;
        dst = prm.q + ((size_t)m * prm.Hq) * D + n0;
      } else if (n0 < (prm.Hq + prm.Hkv) * D) {
        sect = 1;
        dst = prm.kn + ((size_t)m * prm.Hkv) * D + (n0 - prm.Hq * D);
      } else {
        dst = prm.vn + ((size_t)m * prm.Hkv) * D + (n0 - (prm.Hq + prm.Hkv) * D);
      }
      // the first position of each pair the tile touches (uniform branch)
      int slot = 0, t = 0;
      if (sect) {
        const int p_first = m0 / prm.l;
        named_bar_sync(1, kEpi);  // every thread is done with the previous tile's slots
        for (int idx = r; idx < kMaxSlots * (HALF / 2); idx += kEpi) {
          const int sl = idx / (HALF / 2), jp = idx - sl * (HALF / 2);
          const int p = p_first + sl;
          if (p * prm.l < prm.M) {
            const int pos = prm.pos_offset ? prm.pos_offset[p] : prm.C;
            float s0, c0, s1, c1;
            sincosf((float)pos * prm.inv_freq[2 * jp], &s0, &c0);
            sincosf((float)pos * prm.inv_freq[2 * jp + 1], &s1, &c1);
            *reinterpret_cast<float4*>(base + idx * 16) = make_float4(c0, c1, s0, s1);
          }
        }
        named_bar_sync(1, kEpi);
        const int p = m / prm.l;
        slot = p - p_first;
        t = m - p * prm.l;
      }
      if (!failed && !mbar_wait(&bars->acc_full[b], (uint32_t)(tl >> 1) & 1u)) failed = true;
      tc::fence_after_sync();
      const uint32_t acc = tmem + lane_base + b * kBN;
      if (sect) {
        // heads of D columns: chunk c (16 columns) pairs with chunk c + D/32
        const uint8_t* trow = tab + t * (HALF / 2) * 16;
        const uint8_t* brow = base + slot * (HALF / 2) * 16;
#pragma unroll 1
        for (int c = 0; c < kBN / 16; ++c) {
          if ((c % (D / 16)) >= D / 32) continue;  // the second half of a head
          uint32_t xv[16], yv[16];
          tc::ld16(acc + c * 16, xv);
          tc::ld16(acc + (c + D / 32) * 16, yv);
          tc::wait_ld();
          const int j0 = (c % (D / 16)) * 16;  // first frequency of the chunk
          uint32_t xw[8], yw[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int jp = (j0 >> 1) + e;
            const uint4 cs = *reinterpret_cast<const uint4*>(trow + jp * 16);
            const uint4 bs = *reinterpret_cast<const uint4*>(brow + jp * 16);
            const uint64_t tc2 = f2_make(__uint_as_float(cs.x), __uint_as_float(cs.y));
            const uint64_t ts2 = f2_make(__uint_as_float(cs.z), __uint_as_float(cs.w));
            const uint64_t bc2 = f2_make(__uint_as_float(bs.x), __uint_as_float(bs.y));
            const uint64_t bs2 = f2_make(__uint_as_float(bs.z), __uint_as_float(bs.w));
            // angle of position pos0 + t = angle(pos0) + angle(t)
            const uint64_t cc = f2_sub(f2_mul(bc2, tc2), f2_mul(bs2, ts2));
            const uint64_t ss = f2_fma(bs2, tc2, f2_mul(bc2, ts2));
            const uint64_t x = f2_make(__uint_as_float(xv[2 * e]), __uint_as_float(xv[2 * e + 1]));
            const uint64_t y = f2_make(__uint_as_float(yv[2 * e]), __uint_as_float(yv[2 * e + 1]));
            xw[e] = f2_to_bf16x2(f2_sub(f2_mul(x, cc), f2_mul(y, ss)));
            yw[e] = f2_to_bf16x2(f2_fma(y, cc, f2_mul(x, ss)));
          }
          if (m < prm.M) {
            stg16(dst + c * 16, make_uint4(xw[0], xw[1], xw[2], xw[3]));
            stg16(dst + c * 16 + 8, make_uint4(xw[4], xw[5], xw[6], xw[7]));
            stg16(dst + (c + D / 32) * 16, make_uint4(yw[0], yw[1], yw[2], yw[3]));
            stg16(dst + (c + D / 32) * 16 + 8, make_uint4(yw[4], yw[5], yw[6], yw[7]));
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < kBN / 16; ++c) {
          uint32_t v[16];
          tc::ld16(acc + c * 16, v);
          tc::wait_ld();
          if (m < prm.M) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = f2_to_bf16x2(f2_make(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])));
            stg16(dst + c * 16, make_uint4(w[0], w[1], w[2], w[3]));
            stg16(dst + c * 16 + 8, make_uint4(w[4], w[5], w[6], w[7]));
          }
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&bars->acc_empty[b]);
    }
    if (failed && r == 0) report(prm.status, GIST_ATTN_STATUS_TIMEOUT);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 2 * kBN);
  }
}

// Row-major [rows][cols] bf16, tiles of kBK columns x 128 rows, 128-byte swizzle.
int encode_2d(CUtensorMap* m, const void* base, int rows, int cols) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return GIST_ATTN_ERR_LAUNCH;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {kBK, kBM};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GIST_ATTN_OK : GIST_ATTN_ERR_UNSUPPORTED;
}

template <int D>
int launch_gemm_d(GemmParams prm, const void* a, const void* b, cudaStream_t stream) {
  alignas(64) CUtensorMap tm_a, tm_b;
  int rc = encode_2d(&tm_a, a, prm.M, prm.K);
  if (rc != GIST_ATTN_OK) return rc;
  rc = encode_2d(&tm_b, b, prm.N, prm.K);
  if (rc != GIST_ATTN_OK) return rc;
  uint32_t off = kStages * 2 * kTile;
  prm.off_tab = off;
  off += prm.qkv ? (uint32_t)prm.l * (D / 4) * 16 : 0;
  prm.off_base = off;
  off += prm.qkv ? (uint32_t)kMaxSlots * (D / 4) * 16 : 0;
  prm.off_bar = off;
  off += 128;
  const uint32_t bytes = off + 1024;
  if (bytes > (uint32_t)kMaxSmem) return GIST_ATTN_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(gemm_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GIST_ATTN_ERR_LAUNCH;
  const int grid = prm.num_tiles < sms ? prm.num_tiles : sms;
  gemm_kernel<D><<<grid, kThreads, bytes, stream>>>(tm_a, tm_b, prm);
  return cudaGetLastError() == cudaSuccess ? GIST_ATTN_OK : GIST_ATTN_ERR_LAUNCH;
}

int launch_common(GemmParams& prm, const void* a, const void* b, int d, cudaStream_t stream) {
  const int64_t mt = ((int64_t)prm.M + kBM - 1) / kBM;
  prm.ntn = prm.N / kBN;
  if (mt * prm.ntn > 0x7fffffff) return GIST_ATTN_ERR_UNSUPPORTED;
  prm.num_tiles = (int)(mt * prm.ntn);
  if (prm.num_tiles == 0) return GIST_ATTN_OK;
  if (d == 64) return launch_gemm_d<64>(prm, a, b, stream);
  return launch_gemm_d<128>(prm, a, b, stream);
}

}  // namespace

// Sizes this build runs: N a multiple of 128, K a multiple of 8 (16-byte rows
// for TMA), M below 2^31; for the QKV split also head groups that tile N.
bool gemm_fits(int64_t M, int N, int K) {
  return M >= 0 && M < 0x7fffffff && N > 0 && N % kBN == 0 && K > 0 && K % 8 == 0;
}

int launch_qkv_rope(const Problem& pb, const void* x, const void* w, int d_model, void* q,
                    void* kn, void* vn, cudaStream_t stream) {
  GemmParams prm{};
  prm.M = pb.P * pb.l;
  prm.N = (pb.Hq + 2 * pb.Hkv) * pb.d;
  prm.K = d_model;
  if (!gemm_fits((int64_t)pb.P * pb.l, prm.N, prm.K)) return GIST_ATTN_ERR_UNSUPPORTED;
  // every 128-column tile must lie inside one of the q / k / v sections
  if ((pb.Hq * pb.d) % kBN != 0 || (pb.Hkv * pb.d) % kBN != 0) return GIST_ATTN_ERR_UNSUPPORTED;
  // a 128-row tile must touch at most kMaxSlots pairs, and the table hold l rows
  if ((kBM - 1) / pb.l + 2 > kMaxSlots || pb.l > 1024) return GIST_ATTN_ERR_UNSUPPORTED;
  prm.qkv = 1;
  prm.q = static_cast<bf16*>(q);
  prm.kn = static_cast<bf16*>(kn);
  prm.vn = static_cast<bf16*>(vn);
  prm.l = pb.l;
  prm.Hq = pb.Hq;
  prm.Hkv = pb.Hkv;
  prm.d = pb.d;
  prm.C = pb.C;
  prm.pos_offset = pb.pos_offset;
  prm.status = pb.status;
  for (int j = 0; j < 64; ++j) prm.inv_freq[j] = pb.inv_freq[j];
  return launch_common(prm, x, w, pb.d, stream);
}

int launch_out_proj(const Problem& pb, const void* attn, const void* w, int d_model, void* y,
                    cudaStream_t stream) {
  GemmParams prm{};
  prm.M = pb.P * pb.l;
  prm.N = d_model;
  prm.K = pb.Hq * pb.d;
  if (!gemm_fits((int64_t)pb.P * pb.l, prm.N, prm.K)) return GIST_ATTN_ERR_UNSUPPORTED;
  prm.qkv = 0;
  prm.y = static_cast<bf16*>(y);
  prm.status = pb.status;
  prm.l = pb.l;
  return launch_common(prm, attn, w, 64, stream);
}

}  // namespace gattn
