/*
 * gist_attn.h -- C ABI of the GB300 (sm_103a) library for per-layer GQA
 * attention of a short block of new tokens against a read-only cached KV
 * segment.
 *
 * Sources, cited by page title and section:
 *   [Gist page]   "把 item 压成 KV：gist 能不能用在相关性任务上" (liam.page, 2026-10-30)
 *   [Suffix page] icman.com.cn news 64898 (suffix KV-cache reuse and attention-aware
 *                 eviction), numbered sections 1-7
 *   [KV page]     "为什么自回归推理缓存 KV，而不缓存历史 Q？" (mcfzz.com notes)
 *
 * The operation ([Gist page, "在线的一次 attention"]; [KV page, "Reusable-state"]):
 * for every pair p (an (item, query) pair, or a sequence in decode), every
 * query head h and every new token i,
 *
 *     out[p,i,h] = softmax( scale * R(q[p,i,h]) . [K_cached ; R(k_new[p,0..i,g])]^T )
 *                  . [V_cached ; v_new[p,0..i,g]]
 *
 * with g = h / (Hq/Hkv) the KV head of h's group ([Gist page, "收益有多大：存储"]),
 * R the rotate-half RoPE at position pos_offset[p] + i (new keys at their own
 * positions), K_cached/V_cached the rows of p's cached blocks in table order,
 * and nothing written back ([Gist page, "能不能再进一步"]: the cached blocks are
 * read-only and the new tokens' K/V are not stored).
 *
 * Conventions for every entry point:
 *   - Ownership: the caller owns every buffer.  No entry point allocates
 *     memory or keeps state between calls; calls are thread-safe.  (The one
 *     exception, gist_attn_fwd_noalloc, keeps a fixed scratch array of its own.)
 *   - Asynchrony: work is enqueued on `stream` (0 = legacy default stream);
 *     no entry point synchronises the host.
 *   - Pointers are device pointers unless marked "host".  bf16 buffers must be
 *     16-byte aligned, int32 buffers 4-byte aligned.
 *   - Return codes are host-detected and mean nothing was launched:
 *       GIST_ATTN_OK (0), or one of the negative GIST_ATTN_ERR_* codes.
 *   - Device-detected problems are OR-ed into the optional device status word
 *     (dims->status) as GIST_ATTN_STATUS_* bits; the kernel never reads out of
 *     bounds because of them.
 */
#ifndef GIST_ATTN_H
#define GIST_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host return codes. */
#define GIST_ATTN_OK 0
#define GIST_ATTN_ERR_NULL (-1)        /* a required pointer is NULL                    */
#define GIST_ATTN_ERR_DIMS (-2)        /* inconsistent or out-of-range dimensions       */
#define GIST_ATTN_ERR_UNSUPPORTED (-3) /* head_dim / group / sizes this build can't run */
#define GIST_ATTN_ERR_ALIGN (-4)       /* a pointer is not aligned as required          */
#define GIST_ATTN_ERR_LAUNCH (-5)      /* the CUDA launch itself failed                 */
#define GIST_ATTN_ERR_SCRATCH (-6)     /* gist_attn_fwd_noalloc: the call needs more
                                          scratch than the library's fixed array holds */

/* Device status bits (OR-ed into *dims->status). */
#define GIST_ATTN_STATUS_BAD_BLOCK 1 /* a block id was outside [0, num_blocks): that
                                        pair's output rows were written as zeros     */
#define GIST_ATTN_STATUS_TIMEOUT 2   /* a bounded wait on an asynchronous copy gave up;
                                        the affected outputs are unspecified          */
#define GIST_ATTN_STATUS_RANGE 4     /* a row's softmax sum was not finite even in
                                        fp32: a NaN input, or logits or values near the
                                        fp32 limit; that row's outputs are not finite.
                                        (Values past the f16 range alone do not set it:
                                        the kernels that form q.K in f16 recompute the
                                        rows they reach in fp32.)                      */

typedef struct {
  int32_t num_pairs;       /* P >= 0: pairs (or decode sequences) in this call          */
  int32_t n_new;           /* l >= 1: new tokens per pair, EOS included                 */
  int32_t num_q_heads;     /* Hq >= 1                                                    */
  int32_t num_kv_heads;    /* Hkv >= 1, Hq % Hkv == 0; q head h reads KV head h/(Hq/Hkv) */
  int32_t head_dim;        /* d: 64 or 128                                               */
  int32_t block_len;       /* cached positions per pool block (k for a gist item,
                              256 for the paged pool of [Suffix page, §5])               */
  int32_t blocks_per_pair; /* cached blocks per pair: 1 (item gist), 2 (item + query
                              gist, [Gist page, "能不能再进一步"]), T/256 (paged)          */
  int32_t num_blocks;      /* pool extent; every block id must lie in [0, num_blocks)  */
  int32_t num_layers;      /* L: layers held by the pool                                 */
  int32_t layer;           /* the layer this call reads, 0 <= layer < L                  */
  float rope_theta;        /* RoPE base (1e4 in the workloads), > 0                      */
  float softmax_scale;     /* 0 selects 1/sqrt(d) ([KV page, "Reusable-state"])          */
  int32_t* status;         /* optional device int32 status word (may be NULL)            */
  int32_t flags;           /* GIST_ATTN_FLAG_* bits; 0 for the plain operation           */
} gist_attn_dims;

/* dims->flags: q and k_new arrive already rotated at their positions (for example
 * by gist_qkv_rope), so the attention and the pool writers apply no RoPE. */
#define GIST_ATTN_FLAG_PREROTATED 1
/* dims->flags, for tests of the error path only: the paged MHA decode step
 * (gist_attn_fwd with l = 1, equal head counts, 64+ cached rows in 16-row
 * blocks) withholds the copy of its first cached chunk and shortens its
 * bounded waits to 20 ms, so every CTA gives up, waits for the copies it did
 * issue, and reports GIST_ATTN_STATUS_TIMEOUT; the outputs are then
 * unspecified.  Other kernels ignore the flag.  Nothing faults or hangs. */
#define GIST_ATTN_FLAG_TEST_WITHHOLD 2

/*
 * gist_attn_fwd -- one layer of attention for all pairs, one launch on `stream`.
 * Defined by [Gist page, "在线的一次 attention"] (cat of cached and new K/V, new
 * tokens numbered after the cached positions), [Gist page, "能不能再进一步"]
 * (two read-only cached blocks, l = 1) and [KV page, "Reusable-state"] (the
 * decode step, l = 1, over a paged cache read through a block table as in
 * [Suffix page, §6 问题四]).
 *
 *   q          bf16 [P][l][Hq][d], pre-RoPE
 *   k_new      bf16 [P][l][Hkv][d], pre-RoPE
 *   v_new      bf16 [P][l][Hkv][d]
 *   kv_pool    bf16 [num_blocks][L][2][Hkv][block_len][d]; index 0 of the "2"
 *              axis is K (stored already rotated at the positions its producer
 *              chose), 1 is V.  Read-only.
 *   item_ids   int32 [P]: the one cached block of each pair (blocks_per_pair == 1),
 *              or NULL
 *   block_table int32 [P][blocks_per_pair]: cached blocks in key order, or NULL.
 *              Exactly one of item_ids / block_table is non-NULL when the cached
 *              segment is non-empty (blocks_per_pair * block_len > 0).
 *   pos_offset int32 [P]: position of new token 0, or NULL for
 *              blocks_per_pair * block_len (the query follows the cached
 *              segment).  Only pos_offset minus the cached keys' positions
 *              matters ([Gist page, "在线的一次 attention"], RoPE remark).
 *   out        bf16 [P][l][Hq][d], written (fp32 accumulation, round to nearest even)
 *   dims       host pointer to the dimensions above
 * Returns GIST_ATTN_OK or a negative GIST_ATTN_ERR_* code (nothing launched).
 * P == 0 launches nothing and returns GIST_ATTN_OK.
 */
int gist_attn_fwd(const void* q, const void* k_new, const void* v_new, const void* kv_pool,
                  const int32_t* item_ids, const int32_t* block_table, const int32_t* pos_offset,
                  void* out, const gist_attn_dims* dims, cudaStream_t stream);

/*
 * gist_attn_workspace_bytes -- device bytes of the workspace gist_attn_fwd_ws
 * uses for these dimensions, or 0 when they run without one.  Host only.
 * Non-zero for d = 64, n_new >= 2, cached + new keys above the 288 that the
 * single-pass tensor-core kernel holds, and groups of at most 128 heads (cached
 * blocks per pair <= 64), where the staged path applies: 256 * P + 256 * n_new +
 * 2 * (2 * P * (cached + n_new) * Hkv * 64) bytes, each of the four parts
 * rounded up to 256.  Invalid dims return 0.
 */
size_t gist_attn_workspace_bytes(const gist_attn_dims* dims);

/*
 * gist_attn_fwd_ws -- gist_attn_fwd with a caller-provided device workspace
 * (the same definition: [Gist page, "在线的一次 attention"], K = cat(cached K,
 * new K) with the new tokens numbered after the cached positions, causal
 * inside the new block).  Arguments as gist_attn_fwd, plus:
 *   workspace       device pointer, 256-byte aligned, at least
 *                   gist_attn_workspace_bytes(dims) bytes, or NULL
 *   workspace_bytes its size in bytes
 * Where the workspace applies and is large enough, a pre-pass writes each
 * pair's key sequence [cached; new] into it (keys rotated and rounded once to
 * f16, values bf16) with the rotation angles of q, and the long-sequence
 * tensor-core kernel runs on that, rotating q (rounded once to f16) as it
 * loads each tile: two launches on `stream`.  The caller owns the workspace; its
 * contents are scratch, overwritten by every call, and must not be touched
 * until the work on `stream` has finished.  Otherwise (no workspace, too small,
 * misaligned, or shapes without a staged path) the call does exactly what
 * gist_attn_fwd does.  Errors as gist_attn_fwd; a block id outside the pool
 * zeroes that pair's rows and sets GIST_ATTN_STATUS_BAD_BLOCK, a value past the
 * f16 range sets GIST_ATTN_STATUS_RANGE.
 */
int gist_attn_fwd_ws(const void* q, const void* k_new, const void* v_new, const void* kv_pool,
                     const int32_t* item_ids, const int32_t* block_table,
                     const int32_t* pos_offset, void* out, void* workspace, size_t workspace_bytes,
                     const gist_attn_dims* dims, cudaStream_t stream);

/*
 * gist_attn_fwd_noalloc -- gist_attn_fwd_ws without a caller workspace and
 * without any allocation.  The paper has no counterpart: this entry point is
 * for callers that cannot allocate device memory where they call the
 * attention -- a plugin inside a host program that owns all device memory and
 * gives its kernels no workspace, or a latency-critical loop that must not pay
 * the implicit device synchronisation of cudaMalloc / cudaFree.
 *
 * Arguments, result and errors as gist_attn_fwd.  Where gist_attn_fwd_ws would
 * take its staged path, the scratch it needs lives in a fixed device array of
 * GIST_ATTN_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library, reserved on every
 * device that loads the library's device code until the process exits; calls
 * whose gist_attn_workspace_bytes(dims) exceeds it return GIST_ATTN_ERR_SCRATCH
 * and launch nothing.  Shapes without a staged path need no scratch and run
 * exactly as gist_attn_fwd.  No call allocates or frees memory.
 *   - Set-up: the first call on a device that needs scratch looks up the
 *     array's device address (cudaGetSymbolAddress, with the caller's current
 *     device, which must be the device of `stream`); GIST_ATTN_ERR_LAUNCH if
 *     that fails.  Make that first call before any stream capture.
 *   - Sharing: every call on a device uses the same array, and it keeps the
 *     previous call's contents; each call writes every scratch byte it reads,
 *     so nothing has to start at zero.  Calls whose work overlaps on the GPU
 *     (other streams, other host threads) race on the array: order them.
 */
#define GIST_ATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int gist_attn_fwd_noalloc(const void* q, const void* k_new, const void* v_new,
                          const void* kv_pool, const int32_t* item_ids,
                          const int32_t* block_table, const int32_t* pos_offset, void* out,
                          const gist_attn_dims* dims, cudaStream_t stream);

/*
 * gist_attn_fwd_fp8kv -- gist_attn_fwd with the cached segment stored as FP8
 * E4M3 bytes ([Suffix page, §2 and the end of §5]: a 1-byte-per-element KV
 * cache).  The pages give no scale convention; here each (block, layer, K|V,
 * KV head) has one fp32 scale and a cached value is e4m3 * scale.
 *   kv_pool_e4m3 uint8 [num_blocks][L][2][Hkv][block_len][d] (same layout as the
 *                bf16 pool, one byte per element), 16-byte aligned
 *   kv_scale     float [num_blocks][L][2][Hkv], 4-byte aligned
 * Other arguments as gist_attn_fwd.  This build runs blocks of l >= 2 new
 * tokens whose cached rows and new tokens together are at most 288 keys for
 * d = 64 and 128 for d = 128, with at most 128 query heads per KV head (the
 * shapes of gist_attn_fwd's tensor-core prefill), and the decode step (l = 1):
 * equal query and KV head counts with a cache of at least 64 rows in blocks
 * of a multiple of 16 rows (the paged layout); groups of 2..16 query heads
 * with more than 32 cached rows in at most 512 blocks of a multiple of 16 rows
 * (GQA paged); or groups of at most 16 query heads with at most 32 cached rows
 * in blocks of a multiple of 8 rows (the query-gisted layout of [Gist page,
 * "能不能再进一步"]).  Other shapes return GIST_ATTN_ERR_UNSUPPORTED.  Scales
 * must be finite and non-negative.
 */
int gist_attn_fwd_fp8kv(const void* q, const void* k_new, const void* v_new,
                        const void* kv_pool_e4m3, const float* kv_scale,
                        const int32_t* item_ids, const int32_t* block_table,
                        const int32_t* pos_offset, void* out, const gist_attn_dims* dims,
                        cudaStream_t stream);

/*
 * gist_attn_fwd_block_mass -- the decode step (l = 1) of gist_attn_fwd over a
 * paged cache, also writing each cached block's attention mass, the statistic
 * of the attention-aware eviction in [Suffix page, §4 and §5 第三步] (every 64
 * generated tokens the caller averages the weights per history token and marks
 * blocks below 0.3 x the mean; the policy itself is the caller's):
 *   block_mass  float [P][Hq][blocks_per_pair]: the sum of head h's softmax
 *               weights over the rows of the b-th block of p's table.  The new
 *               token's own weight is 1 - sum_b block_mass[p][h][b].
 * Other arguments as gist_attn_fwd (block_table required).  This build runs
 * groups of 1..16 query heads per KV head over blocks of a multiple of 16 rows:
 * equal head counts with 64..8192 cached rows, or 2..16 heads per KV head with
 * 33..8192 cached rows in at most 512 blocks; other shapes return
 * GIST_ATTN_ERR_UNSUPPORTED.
 */
int gist_attn_fwd_block_mass(const void* q, const void* k_new, const void* v_new,
                             const void* kv_pool, const int32_t* block_table,
                             const int32_t* pos_offset, void* out, float* block_mass,
                             const gist_attn_dims* dims, cudaStream_t stream);

/*
 * gist_kv_append -- writes one new token per sequence into the paged cache at
 * `layer` ([KV page, "Reusable-state"]: K_{<=t} = [K_{<t}; k_t], the new K/V
 * are appended to every layer's cache).  For sequence p and KV head g:
 *   kv_pool[block_table[p][slot[p] / block_len]][layer][0][g][slot[p] % block_len]
 *       = bf16(R(k_new[p][0][g]))  (RoPE at pos_offset[p], or at slot[p] when NULL;
 *                                   rounded to nearest even)
 *   ... [1][g][same row] = v_new[p][0][g]
 *   k_new, v_new bf16 [P][1][Hkv][d]; slot int32 [P]; kv_pool is written.
 * dims: n_new must be 1 and the table non-empty (GIST_ATTN_ERR_DIMS otherwise).
 * A slot outside [0, blocks_per_pair * block_len) or an out-of-range block id
 * skips that sequence and sets GIST_ATTN_STATUS_BAD_BLOCK.
 */
int gist_kv_append(const void* k_new, const void* v_new, void* kv_pool,
                   const int32_t* block_table, const int32_t* slot, const int32_t* pos_offset,
                   const gist_attn_dims* dims, cudaStream_t stream);

/*
 * gist_attn_fwd_gist_mask -- gist_attn_fwd under the gist mask of
 * [Gist page, "论文做了什么"] (the ordinary causal mask with the block
 * (tokens after the gist) x (tokens before it) removed).  Keys of pair p are
 * numbered kappa = 0 .. C + l - 1 over [cached; new]; the prompt is
 * kappa < gist_start[p], the gist the next gist_len keys.  A token whose own
 * index C + i is at least gist_start[p] + gist_len sees only the keys
 * gist_start[p] <= kappa <= C + i; every other token sees kappa <= C + i.
 * With an empty cache and the new tokens [prompt; gist; rest] this is the
 * training-layout forward of whole sequences (sequences of different lengths
 * right-padded to l, their own gist_start each); over [prompt; gist] alone it is
 * the plain causal pass of the offline compression ([Gist page, "在线的一次
 * attention"]: the item is forwarded once, offline).
 *   gist_start int32 [P], device, required; a negative value is taken as 0
 *   gist_len   host int >= 0 (GIST_ATTN_ERR_DIMS otherwise)
 * Other arguments as gist_attn_fwd.  Runs on the streaming kernel: any cache
 * length and l; groups of at most 64 query heads per KV head, and at most 4096
 * cached blocks per pair (GIST_ATTN_ERR_UNSUPPORTED otherwise).
 */
int gist_attn_fwd_gist_mask(const void* q, const void* k_new, const void* v_new,
                            const void* kv_pool, const int32_t* item_ids,
                            const int32_t* block_table, const int32_t* pos_offset,
                            const int32_t* gist_start, int gist_len, void* out,
                            const gist_attn_dims* dims, cudaStream_t stream);

/*
 * gist_kv_store -- writes compressed items into the pool ([Gist page,
 * "论文做了什么"]: after the offline pass over [prompt; gist], each layer keeps
 * the K/V at the k gist positions as the item's cache entry).  dims: n_new = l,
 * the sequence length; block_len = k, the gist length (1 <= k <= l);
 * blocks_per_pair = 1; num_blocks, num_layers, layer as usual (GIST_ATTN_ERR_DIMS
 * otherwise).  For pair p, KV head g and t < k:
 *   kv_pool[item_ids[p]][layer][0][g][t] = bf16(R(k_new[p][first_row[p] + t][g]))
 *       (RoPE at store_pos[p] + t, or at t when store_pos is NULL, i.e. the
 *        online layout where the query follows the gist; rounded to nearest even)
 *   kv_pool[item_ids[p]][layer][1][g][t] = v_new[p][first_row[p] + t][g]
 *   k_new, v_new bf16 [P][l][Hkv][d] (pre-RoPE keys, as gist_attn_fwd takes them)
 *   item_ids, first_row int32 [P]; store_pos int32 [P] or NULL; kv_pool is written.
 * A pair whose rows leave [0, l) or whose block id is out of range is skipped and
 * sets GIST_ATTN_STATUS_BAD_BLOCK.  Two pairs naming the same block race.
 */
int gist_kv_store(const void* k_new, const void* v_new, void* kv_pool, const int32_t* item_ids,
                  const int32_t* first_row, const int32_t* store_pos, const gist_attn_dims* dims,
                  cudaStream_t stream);

/*
 * gist_qkv_rope -- the QKV projection of the new tokens with RoPE in its
 * epilogue, the fusion before the attention ([Gist page, "在线的一次 attention"]:
 * per layer X is projected to Q, K, V, then attends).  For every new token row
 * m = p*l + i:
 *   [q | k | v][m] = x[m] . w_qkv^T   (fp32 accumulation), then q and k heads are
 *   rotated at position pos_offset[p] + i (NULL: blocks_per_pair*block_len + i)
 *   from the fp32 values and rounded once to bf16 (nearest even).
 *   x      bf16 [P][l][d_model], 16-byte aligned, d_model a multiple of 8
 *   w_qkv  bf16 [(Hq + 2 Hkv) d][d_model]: rows are q heads, then k heads, then v heads
 *   q      bf16 [P][l][Hq][d];  k_new, v_new bf16 [P][l][Hkv][d]  (written)
 * Feed the results to gist_attn_fwd with GIST_ATTN_FLAG_PREROTATED.  This build
 * needs Hq*d and Hkv*d multiples of 128, l >= 22 (a 128-row tile spans at most
 * 8 pairs) and l <= 1904 for d = 64, l <= 936 for d = 128 (the table of token
 * angles sits in shared memory), else GIST_ATTN_ERR_UNSUPPORTED.
 */
int gist_qkv_rope(const void* x, const void* w_qkv, const int32_t* pos_offset, void* q,
                  void* k_new, void* v_new, int d_model, const gist_attn_dims* dims,
                  cudaStream_t stream);

/*
 * gist_out_proj -- the output projection after the attention: for every row
 * m < P*l, y[m] = attn_out[m] . w_o^T (fp32 accumulation, bf16 out).
 *   attn_out bf16 [P][l][Hq][d] (gist_attn_fwd's out), w_o bf16 [d_model][Hq d],
 *   y bf16 [P][l][d_model] (written).  d_model must be a multiple of 128 and Hq*d of 8.
 */
int gist_out_proj(const void* attn_out, const void* w_o, void* y, int d_model,
                  const gist_attn_dims* dims, cudaStream_t stream);

/*
 * gist_attn_gather_debug -- copies, bit for bit, the cached rows each pair
 * reads, through the same device gather routine the attention kernels use
 * ([Gist page, "在线的一次 attention"]: cache[item].K[layer], .V[layer]).
 *   dst  bf16 [P][Hkv][2][C][d], C = blocks_per_pair * block_len:
 *        dst[p][g][kv][c] = kv_pool[block(p, c / block_len)][layer][kv][g][c % block_len]
 * A pair with an out-of-range block id gets zero rows and sets
 * GIST_ATTN_STATUS_BAD_BLOCK.  q/k_new/v_new are not read.
 */
int gist_attn_gather_debug(const void* kv_pool, const int32_t* item_ids,
                           const int32_t* block_table, void* dst, const gist_attn_dims* dims,
                           cudaStream_t stream);

/*
 * Cache byte counts, host only, no device work.
 * [Gist page, "先看复用结构" / "收益有多大：存储"]: one position holds
 * 2 * L * Hkv * d numbers of elem_bytes bytes each; a compressed item holds k
 * positions ([Gist page, "在线的一次 attention"]).  [KV page, "Memory"]:
 * M_KV = 2 * B * L * T * Hkv * d * elem_bytes.  Return 0 for a negative argument.
 */
size_t gist_kv_bytes_per_position(int L, int Hkv, int d, int elem_bytes);
size_t gist_kv_bytes_per_item(int L, int Hkv, int d, int k, int elem_bytes);
size_t gist_kv_bytes_batch(int B, int L, int T, int Hkv, int d, int elem_bytes);

/*
 * Text for a return code (negative) or a device status word (>= 0, bits OR-ed).
 * The string is static; the caller must not free it.
 */
const char* gist_attn_status_string(int status);

/*
 * gist_attn_route -- which kernel an entry point runs for these dimensions, as
 * a host-only query: nothing is read from device memory and nothing is
 * launched.  The answer comes from the same function the entry point's own
 * dispatch uses, so a caller (or a test) can see which path a shape takes
 * before it provides any buffer.  The pages define no such call; it exposes
 * how this library splits the attention of [Gist page, "在线的一次 attention"]
 * and the decode step of [KV page, "Reusable-state"] across its kernels.
 *   entry  one of GIST_ATTN_ENTRY_*; GIST_ATTN_ENTRY_FWD_WS answers for
 *          gist_attn_fwd_ws (and gist_attn_fwd_noalloc) given a workspace of
 *          at least gist_attn_workspace_bytes(dims) bytes
 *   dims   as for that entry point (the gist-mask entry with gist_len 0)
 * Returns one of GIST_ATTN_ROUTE_* (>= 0; GIST_ATTN_ROUTE_NONE when num_pairs
 * is 0), the GIST_ATTN_ERR_* code the entry point's dimension checks return,
 * or GIST_ATTN_ERR_UNSUPPORTED when no kernel takes the shape (or `entry` is
 * not one of the values below).
 */
#define GIST_ATTN_ENTRY_FWD 0        /* gist_attn_fwd                               */
#define GIST_ATTN_ENTRY_FWD_WS 1     /* gist_attn_fwd_ws / _noalloc with workspace  */
#define GIST_ATTN_ENTRY_FP8KV 2      /* gist_attn_fwd_fp8kv                         */
#define GIST_ATTN_ENTRY_BLOCK_MASS 3 /* gist_attn_fwd_block_mass                    */
#define GIST_ATTN_ENTRY_GIST_MASK 4  /* gist_attn_fwd_gist_mask                     */

#define GIST_ATTN_ROUTE_NONE 0           /* nothing to launch (num_pairs == 0)          */
#define GIST_ATTN_ROUTE_PREFILL_TC 1     /* tcgen05 prefill, a tile's keys in one pass  */
#define GIST_ATTN_ROUTE_PREFILL_LONG 2   /* tcgen05 prefill over 128-key blocks         */
#define GIST_ATTN_ROUTE_PREFILL_STREAM 3 /* streaming mma.sync prefill, any length      */
#define GIST_ATTN_ROUTE_STAGED 4         /* staging pre-pass, then the 128-key blocks   */
#define GIST_ATTN_ROUTE_DECODE_LONG 5    /* l = 1, one head per KV head, long cache     */
#define GIST_ATTN_ROUTE_DECODE_SHORT 6   /* l = 1, cache of at most 32 keys             */
#define GIST_ATTN_ROUTE_DECODE_GQA 7     /* l = 1, 2..16 heads per KV head, longer cache */
#define GIST_ATTN_ROUTE_DECODE 8         /* l = 1, the other shapes (CUDA cores)        */

int gist_attn_route(int entry, const gist_attn_dims* dims);

#ifdef __cplusplus
}
#endif

#endif /* GIST_ATTN_H */
