// exact.cuh -- one query row of the attention in fp32 on the CUDA cores, read
// straight from the call's own inputs: the fallback of the kernels that form
// q . K in f16.
//
// The operation is the one of [Gist page, "在线的一次 attention"] (keys are the
// pair's cached rows in table order, then its new keys rotated at their
// positions, causal): out = softmax(scale R(q) . K^T) V over the visible keys
// [lo, hi) of the [cached; new] numbering.  The tensor-core kernels round
// rotated q and the keys to f16 (11 significant bits) for the product; a value
// past the f16 range (|x| >= 65520, a legal bf16 value) becomes inf there and
// the row's softmax sum comes out non-finite.  Such a row is recomputed here:
// q and the new keys are rotated in fp32 with angles reduced in double, logits
// and weights in fp32 (online maximum), fp32 accumulation.  Rows that never see
// such a value never come here; the cost of a row is O((hi - lo) d) plus one
// sine/cosine per new key and frequency.
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上".
#pragma once

#include "common.cuh"

namespace gattn {

// Rows whose largest logit (log2 units, scale applied) exceeds this are also
// recomputed here by the kernels that round q and the keys to f16 for q.K: the
// rounding puts an error of about 2^-12 |q| |k| scale on every logit, and large
// logits come with large norms, so past ~20 (about 14 nats) that error nears
// the parity bound of the outputs.  Ordinary rows sit far below it.
constexpr float kExactLogit = 20.f;

// The call's inputs as the C ABI received them.
struct ExactInputs {
  const bf16* q;      // [P][l][Hq][d]
  const bf16* k_new;  // [P][l][Hkv][d]
  const bf16* v_new;  // [P][l][Hkv][d]
  PoolView pv;        // cached rows: blocks_per_pair x block_len = C per pair
  const int32_t* pos_offset;  // [P] or nullptr (new token 0 at position C)
  int l, Hq, Hkv, C;
  int rotate;        // 0: q and k_new arrive rotated
  float scale_log2;  // softmax scale x log2(e)
  double theta[64];  // RoPE frequencies rope_theta^(-2j/d), j < d/2
  // FP8 pool: one fp32 scale per (block, layer, K|V, KV head), the pool's rows
  // E4M3 bytes at the same element offsets; null for a bf16 pool
  const float* kv_scale;
};

// Two E4M3 bytes (the low 16 bits) -> an f16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3_pair_to_f16x2(uint32_t v16) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((unsigned short)v16));
  return r;
}
// An f16 pair -> fp32 (low half first).
__device__ __forceinline__ void f16x2_to_floats(uint32_t h, float& lo, float& hi) {
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
}
// One E4M3 byte -> fp32, exactly.
__device__ __forceinline__ float e4m3_to_float(uint8_t b) {
  float lo, hi;
  f16x2_to_floats(e4m3_pair_to_f16x2(b), lo, hi);
  return lo;
}

// Rotates v at position `pos`: each pair (v[j], v[j + d/2]) by pos * theta_j.
template <int D>
__device__ __forceinline__ void exact_rotate(float (&v)[D], long long pos, const double* theta) {
#pragma unroll 1
  for (int j = 0; j < D / 2; ++j) {
    float s, c;
    sincosf(rope_reduce(pos, theta[j]), &s, &c);
    const float x = v[j], y = v[j + D / 2];
    v[j] = x * c - y * s;
    v[j + D / 2] = y * c + x * s;
  }
}

template <int D>
__device__ __forceinline__ void exact_load_row(float (&v)[D], const bf16* src) {
#pragma unroll 1
  for (int j = 0; j < D; ++j) v[j] = __bfloat162float(src[j]);
}
// A cached row of an FP8 pool (E4M3 bytes), dequantised by its scale.
template <int D>
__device__ __forceinline__ void exact_load_row8(float (&v)[D], const uint8_t* src, float scale) {
#pragma unroll 1
  for (int j = 0; j < D; ++j) v[j] = e4m3_to_float(src[j]) * scale;
}

// Output columns col(i) = c0 + (i / 2) * cstep + (i % 2), i < NC, of row
// (pair p, new token t, query head hq), normalised, into o.  Keys [lo, hi).
// Returns false if the row's sum is not finite (an fp32 overflow or a NaN
// input), in which case o holds what the arithmetic gave.
template <int D, int NC>
__device__ __forceinline__ bool exact_row(const ExactInputs& in, int p, int t, int hq, int lo, int hi,
                                       int c0, int cstep, float (&o)[NC]) {
  const int G = in.Hq / in.Hkv, g = hq / G;
  const long long pos0 = in.pos_offset ? (long long)in.pos_offset[p] : (long long)in.C;
  float qr[D], kr[D];
  exact_load_row<D>(qr, in.q + (((size_t)p * in.l + t) * in.Hq + hq) * D);
  if (in.rotate) exact_rotate<D>(qr, pos0 + t, in.theta);
  float m = -INFINITY, lsum = 0.f;
  // (loops over o stay rolled: the accumulator lives in local memory, so this
  // rarely taken path adds no register pressure to the kernel around it)
#pragma unroll 1
  for (int i = 0; i < NC; ++i) o[i] = 0.f;
#pragma unroll 1
  for (int kappa = lo; kappa < hi; ++kappa) {
    const bf16 *krow, *vrow;
    const uint8_t* vrow8 = nullptr;  // FP8 pool: the cached value row's bytes
    float vsc = 1.f;
    if (kappa < in.C) {
      const int b = kappa / in.pv.block_len, r = kappa - b * in.pv.block_len;
      const int32_t blk = pool_block_id(in.pv, p, b);
      krow = pool_row(in.pv, blk, g, 0, r);
      vrow = pool_row(in.pv, blk, g, 1, r);
      if (in.kv_scale) {
        const uint8_t* base8 = reinterpret_cast<const uint8_t*>(in.pv.pool);
        const int64_t si = (((int64_t)blk * in.pv.num_layers + in.pv.layer) * 2) * in.Hkv + g;
        exact_load_row8<D>(kr, base8 + (krow - in.pv.pool), in.kv_scale[si]);
        vrow8 = base8 + (vrow - in.pv.pool);
        vsc = in.kv_scale[si + in.Hkv];
      } else {
        exact_load_row<D>(kr, krow);
      }
    } else {
      const int i = kappa - in.C;
      const size_t o_new = (((size_t)p * in.l + i) * in.Hkv + g) * D;
      krow = in.k_new + o_new;
      vrow = in.v_new + o_new;
      exact_load_row<D>(kr, krow);
      if (in.rotate) exact_rotate<D>(kr, pos0 + i, in.theta);
    }
    float s = 0.f;
#pragma unroll 1
    for (int j = 0; j < D; ++j) s = fmaf(qr[j], kr[j], s);
    s *= in.scale_log2;
    const float mn = fmaxf(m, s);
    const float al = m == -INFINITY ? 0.f : exp2f(m - mn);
    const float pk = exp2f(s - mn);
    lsum = lsum * al + pk;
#pragma unroll 1
    for (int i = 0; i < NC; ++i) {
      const int col = c0 + (i >> 1) * cstep + (i & 1);
      const float v = vrow8 ? e4m3_to_float(vrow8[col]) * vsc : __bfloat162float(vrow[col]);
      o[i] = o[i] * al + pk * v;
    }
    m = mn;
  }
  const float inv = 1.f / lsum;
#pragma unroll 1
  for (int i = 0; i < NC; ++i) o[i] *= inv;
  return lsum <= 3.0e38f && lsum > 0.f;
}

// Whether a bf16 row of D elements holds a NaN or an infinity.
template <int D>
__device__ __forceinline__ bool row_not_finite(const bf16* row) {
  bool bad = false;
#pragma unroll 1
  for (int c = 0; c < D / 8; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + 8 * c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      bad |= (w[e] & 0x7f80u) == 0x7f80u || (w[e] & 0x7f800000u) == 0x7f800000u;
  }
  return bad;
}

// The repair step of a kernel whose rows came out non-finite: every output row
// of (pair p, KV head g, new tokens [t_begin, t_end)) that holds a NaN or an
// infinity is recomputed in fp32 and written back.  The caller's stores of those
// rows must be complete and visible to this thread.  Threads tid, tid +
// nthreads, ... take the rows.  Keys: the cached rows, then new keys 0..t.
template <int D>
__device__ __forceinline__ void exact_repair_rows(const ExactInputs& in, bf16* out, int p, int g,
                                               int t_begin, int t_end, int tid, int nthreads,
                                               int32_t* status) {
  const int G = in.Hq / in.Hkv;
  for (int idx = tid; idx < (t_end - t_begin) * G; idx += nthreads) {
    const int t = t_begin + idx / G, hq = g * G + idx % G;
    bf16* row = out + (((size_t)p * in.l + t) * in.Hq + hq) * D;
    if (!row_not_finite<D>(row)) continue;
    float o[D];
    if (!exact_row<D, D>(in, p, t, hq, 0, in.C + t + 1, 0, 2, o)) report(status, GIST_ATTN_STATUS_RANGE);
#pragma unroll 1
    for (int c = 0; c < D / 8; ++c)
      *reinterpret_cast<uint4*>(row + 8 * c) =
          make_uint4(float2_to_bf16x2(o[8 * c], o[8 * c + 1]), float2_to_bf16x2(o[8 * c + 2], o[8 * c + 3]),
                     float2_to_bf16x2(o[8 * c + 4], o[8 * c + 5]), float2_to_bf16x2(o[8 * c + 6], o[8 * c + 7]));
  }
}

// Orders this thread's completed bulk (TMA) stores to global memory before its
// later generic-proxy accesses (and, after a barrier, other threads').
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The call's inputs and RoPE frequencies, from the host's problem description.
template <typename Pb>
inline void exact_inputs_from(ExactInputs& e, const Pb& pb) {
  e.q = static_cast<const bf16*>(pb.q);
  e.k_new = static_cast<const bf16*>(pb.k_new);
  e.v_new = static_cast<const bf16*>(pb.v_new);
  e.pv = PoolView{static_cast<const bf16*>(pb.kv_pool), pb.item_ids, pb.block_table,
                  pb.blocks_per_pair, pb.block_len, pb.num_blocks, pb.L, pb.layer, pb.Hkv, pb.d};
  e.pos_offset = pb.pos_offset;
  e.l = pb.l;
  e.Hq = pb.Hq;
  e.Hkv = pb.Hkv;
  e.C = pb.C;
  e.rotate = (pb.flags & GIST_ATTN_FLAG_PREROTATED) ? 0 : 1;
  e.scale_log2 = pb.scale_log2;
  for (int j = 0; j < 64; ++j) e.theta[j] = pb.inv_freq_d[j];
  e.kv_scale = nullptr;
}

}  // namespace gattn
