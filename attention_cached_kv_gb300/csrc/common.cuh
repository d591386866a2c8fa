// common.cuh -- device helpers shared by the attention kernels (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA tensor copies, cp.async, ldmatrix and
// the bf16 tensor-core MMA, the 128-byte shared-memory swizzle, and the one
// routine that turns (pair, cached key) into a pool address -- the gather of
// [Gist page, "在线的一次 attention"] (cache[item].K[layer]) and of the block
// table of [Suffix page, §6 问题四] (logical block -> physical block).
//
// Pages: [Gist page] "把 item 压成 KV：gist 能不能用在相关性任务上";
//        [Suffix page] icman.com.cn news 64898.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver is reached at run time)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gist_attn.h"

namespace gattn {

using bf16 = __nv_bfloat16;

// Every spin on an asynchronous copy gives up after this long and reports
// GIST_ATTN_STATUS_TIMEOUT instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// ------------------------------------------------------------ addresses ---
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Byte offset of 16-byte chunk `chunk` (0..7) of 128-byte row `row` inside a
// panel laid out with the 128-byte swizzle (chunk index XOR row mod 8).  The
// panel base must be 1024-byte aligned; this is the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B and makes ldmatrix conflict-free.
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// ------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(200000u)  // may sleep up to 0.2 ms per try
      : "memory");
  return done != 0;
}
// Waits for the phase with parity `parity` to complete; false after limit_ns
// (kWaitLimitNs unless given).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Plain arrive (count 1) on an mbarrier.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Named barrier 1 among the first `n` threads (a warp-multiple) of the CTA.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Same, returning whether any participant passed `pred` = true.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %3, 0;\n\t"
      "bar.red.or.pred q, %1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(n), "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------ TMA ---
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// 5-D tiled load into shared memory, completing bytes on `bar`.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(c4)
      : "memory");
}
// 2-D tiled load into shared memory, completing bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
// 5-D tiled store from shared memory (elements outside the tensor are dropped).
__device__ __forceinline__ void tma_store_5d(const CUtensorMap* m, uint32_t src, int c0, int c1,
                                             int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group"
      " [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until the shared-memory sources of all committed bulk stores were read.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until all committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tensor core) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------- cp.async ---
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// Waits until at most `n` of this thread's most recent cp.async groups are pending.
template <int n>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory");
}

__device__ __forceinline__ uint4 ldg16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void stg16(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void sts16(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// -------------------------------------------------- ldmatrix / mma.sync ---
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------ bf16 pairs ---
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
// Round to nearest even; `lo` lands in the low half (the lower address).
__device__ __forceinline__ uint32_t float2_to_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------- packed fp32 pairs ---
// Two fp32 values in one 64-bit register; sm_100+ executes f32x2 add/mul/fma
// as one instruction.
__device__ __forceinline__ uint64_t f2_make(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// bf16 pair (low half = first element) -> fp32 pair
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t v) {
  return f2_make(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
// fp32 pair -> bf16 pair, round to nearest even
__device__ __forceinline__ uint32_t f2_to_bf16x2(uint64_t v) {
  float a, b;
  f2_split(v, a, b);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
// Splits an fp32 pair x into hi + lo with hi = x truncated to bf16 (exact in
// fp32, returned packed) and lo = bf16(x - hi): hi + lo carries x to ~16 bits.
__device__ __forceinline__ void f2_split_bf16(uint64_t x, uint32_t& hi_bf, uint32_t& lo_bf) {
  float a, b;
  f2_split(x, a, b);
  const uint32_t ua = __float_as_uint(a) & 0xffff0000u, ub = __float_as_uint(b) & 0xffff0000u;
  hi_bf = __byte_perm(ua, ub, 0x7632);
  lo_bf = f2_to_bf16x2(f2_sub(x, f2_make(__uint_as_float(ua), __uint_as_float(ub))));
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// ----------------------------------------------------------- the gather ---
// The pool is [num_blocks][L][2][Hkv][block_len][d] bf16.
struct PoolView {
  const bf16* pool;
  const int32_t* item_ids;     // [P] or nullptr
  const int32_t* block_table;  // [P][blocks_per_pair] or nullptr
  int32_t blocks_per_pair, block_len, num_blocks, num_layers, layer, num_kv_heads, head_dim;
};

// Block id of pair p's b-th cached block (unchecked).
__device__ __forceinline__ int32_t pool_block_id(const PoolView& v, int p, int b) {
  return v.block_table ? v.block_table[(int64_t)p * v.blocks_per_pair + b] : v.item_ids[p];
}
__device__ __forceinline__ bool pool_block_ok(const PoolView& v, int32_t blk) {
  return blk >= 0 && blk < v.num_blocks;
}
// First element of row t (0 <= t < block_len) of physical block `blk`, for KV
// head g, K (kv = 0) or V (kv = 1), at the layer the view reads.  `blk` must
// have passed pool_block_ok.
__device__ __forceinline__ const bf16* pool_row(const PoolView& v, int32_t blk, int g, int kv,
                                                int t) {
  int64_t r = (int64_t)blk * v.num_layers + v.layer;
  r = (r * 2 + kv) * v.num_kv_heads + g;
  r = r * v.block_len + t;
  return v.pool + r * v.head_dim;
}

// ------------------------------------------------------------ RoPE angle ---
// pos * theta reduced to [-pi, pi]: the product is formed in double (one
// rounding, at most 2^-53 |pos theta| off) and 2 pi is subtracted in two parts
// (the double nearest 2 pi and the remainder), so the angle stays accurate for
// every int32 position; an fp32 product drifts by about |pos theta| 2^-24.
__device__ __forceinline__ float rope_reduce(long long pos, double theta) {
  const double a = (double)pos * theta;
  const double k = rint(a * 0.15915494309189535);  // 1 / (2 pi)
  double r = fma(-k, 6.283185307179586, a);         // 2 pi rounded to double
  r = fma(-k, 2.4492935982947064e-16, r);           // 2 pi minus that
  return (float)r;
}

__device__ __forceinline__ void report(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace gattn
