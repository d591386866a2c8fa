// frag.cuh -- helpers of the mma.sync kernels that take the query heads as the
// N dimension of S^T = K q^T (the short and the long GQA decode): 16-bit MMA,
// in-register 8x8 transposes, E4M3 / f16 conversions, the query's B fragments
// (rotated, scaled, split into hi + lo), and the 2-D tensor maps they load with.
//
// Fragment layouts (PTX m16n8k16): with g8 = lane / 4 and t4 = lane % 4, an A
// register holds row g8 (or g8 + 8), columns 2 t4 and 2 t4 + 1 (or + 8); a B
// register holds rows (k) 2 t4, 2 t4 + 1 (or + 8) of column g8; a C fragment
// holds rows g8 and g8 + 8, columns 2 t4 and 2 t4 + 1.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace gattn {

template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}
// Transposes an 8x8 matrix of 16-bit elements held as one row pair per lane
// (row lane/4, columns 2(lane%4) and +1) into the same layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v16) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)v16));
  return h;
}
// fp32 pair -> f16 pair, round to nearest even (first element in the low half)
__device__ __forceinline__ uint32_t f2_to_f16x2(uint64_t v) {
  float a, b;
  f2_split(v, a, b);
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
__device__ __forceinline__ uint64_t f16x2_to_f2(uint32_t h) {
  float a, b;
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
      : "=f"(a), "=f"(b)
      : "r"(h));
  return f2_make(a, b);
}
// Splits an fp32 pair into f16 hi + lo: hi = f16(x), lo = f16(x - hi).
__device__ __forceinline__ void f2_split_f16(uint64_t x, uint32_t& hi, uint32_t& lo) {
  hi = f2_to_f16x2(x);
  lo = f2_to_f16x2(f2_sub(x, f16x2_to_f2(hi)));
}
// A pair of weights as the 16-bit operand type of P V.
template <bool F16>
__device__ __forceinline__ uint32_t pack_p(float a, float b) {
  if constexpr (F16) return f2_to_f16x2(f2_make(a, b));
  return float2_to_bf16x2(a, b);
}

// 2-D tiled store from shared memory (rows outside the tensor are dropped).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}

// The query's B fragments for one 8-head tile, from its rows in shared memory
// (128-byte swizzle, q_panel bytes per 64-column panel, tile rows hn*8..+7):
// lane gets head row hn*8 + g8, elements d = 16 ks + 8 r + 2 t4 (+1) in
// register [ks][r].  Each element pair (d, d + D/2) is rotated in fp32 by the
// angles cs_of(ks, r) returns for this lane's frequencies j = 16 ks + 8 r + 2 t4
// and j + 1: (c_j, s_j, c_j+1, s_j+1) x scale,
// then split into hi + lo (bf16, or f16 after dividing by the power of two
// *qf so the tile's heads fit f16).  The unrotated query is returned too, for
// the new key's logit: as the raw bf16 B fragments qr, and as the fp32 pairs
// (x, y) = (d, d + D/2).
template <int D, bool F16, class CS>
__device__ __forceinline__ void q_fragments(uint32_t qtile, uint32_t q_panel, int hn, CS cs_of,
                                            uint32_t (&qh)[D / 16][2], uint32_t (&ql)[D / 16][2],
                                            uint32_t (&qr)[D / 16][2], uint64_t (&rx)[D / 16],
                                            uint64_t (&ry)[D / 16], float& qf) {
  constexpr int KS = D / 16, HK = KS / 2;
  const int lane = threadIdx.x & 31;
  uint32_t qb[KS][2];
#pragma unroll
  for (int ks = 0; ks < KS; ks += 2) {
    // matrices (k-step ks: d 0-7, 8-15), (ks + 1: d 0-7, 8-15)
    const int c8 = 2 * ks + (lane >> 3);
    uint32_t r4[4];
    ldsm_x4(qtile + (c8 >> 3) * q_panel + swz128(hn * 8 + (lane & 7), c8 & 7), r4);
    qb[ks][0] = r4[0];
    qb[ks][1] = r4[1];
    qb[ks + 1][0] = r4[2];
    qb[ks + 1][1] = r4[3];
  }
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    qr[ks][0] = qb[ks][0];
    qr[ks][1] = qb[ks][1];
  }
  uint64_t qx[KS], qy[KS];
#pragma unroll
  for (int ks = 0; ks < HK; ++ks) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float4 cs = cs_of(ks, r);
      const uint64_t c = f2_make(cs.x, cs.z), sn = f2_make(cs.y, cs.w);
      const uint64_t x = bf16x2_to_f2(qb[ks][r]), y = bf16x2_to_f2(qb[ks + HK][r]);
      rx[2 * ks + r] = x;
      ry[2 * ks + r] = y;
      qx[2 * ks + r] = f2_sub(f2_mul(x, c), f2_mul(y, sn));
      qy[2 * ks + r] = f2_fma(y, c, f2_mul(x, sn));
    }
  }
  if constexpr (F16) {
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      float a0, a1, b0, b1;
      f2_split(qx[i], a0, a1);
      f2_split(qy[i], b0, b1);
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(b0), fabsf(b1))));
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // e = floor(log2 mx) - 13 for mx >= 2^14 (mx is finite and normal there)
    const int e = mx >= 16384.f ? (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127 - 13 : 0;
    qf = __uint_as_float((uint32_t)(127 + e) << 23);
    const float f = __uint_as_float((uint32_t)(127 - e) << 23);
    const uint64_t f2 = f2_make(f, f);
#pragma unroll
    for (int ks = 0; ks < HK; ++ks)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        f2_split_f16(f2_mul(qx[2 * ks + r], f2), qh[ks][r], ql[ks][r]);
        f2_split_f16(f2_mul(qy[2 * ks + r], f2), qh[ks + HK][r], ql[ks + HK][r]);
      }
  } else {
    qf = 1.f;
#pragma unroll
    for (int ks = 0; ks < HK; ++ks)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        f2_split_bf16(qx[2 * ks + r], qh[ks][r], ql[ks][r]);
        f2_split_bf16(qy[2 * ks + r], qh[ks + HK][r], ql[ks + HK][r]);
      }
  }
}

// [rows][cols] 2-D view of a row-major array, boxes of {box_cols, box_rows},
// 128-byte swizzle (bf16, 64 columns) or none.
inline int encode_2d(CUtensorMap* m, const void* base, CUtensorMapDataType type, int elem_bytes,
              int64_t rows, int cols, int box_cols, int box_rows, bool swizzle) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return GIST_ATTN_ERR_LAUNCH;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * elem_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GIST_ATTN_OK : GIST_ATTN_ERR_UNSUPPORTED;
}

}  // namespace gattn
