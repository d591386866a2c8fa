// noalloc.cu -- gist_attn_fwd_noalloc: the staged path of gist_attn_fwd_ws with
// its scratch held in a fixed device array that belongs to the library, so the
// caller passes no workspace and nothing is allocated on any call.
//
// Who needs this: a caller that cannot allocate device memory at the point of
// the call -- a plugin inside a host program that owns every device allocation
// and hands its kernels no workspace, or a latency-critical loop in which the
// implicit device synchronisation of cudaMalloc / cudaFree is not acceptable.
// Such a caller still owns q, k_new, v_new, the pool, the index arrays and out.
//
// The array `g_stage_scratch` below is a file-scope __device__ variable: every
// device on which the library's device code is loaded reserves it until the
// process exits.  In host code its name is only a host-side stand-in, not a
// device address, so the host looks up the real address once per device with
// cudaGetSymbolAddress (with that device current) and passes that pointer on.
// The paper has no counterpart to this entry point; it is a deployment aid.
#include <mutex>

#include "gist_attn.h"

namespace {

constexpr size_t kStaticScratchBytes = GIST_ATTN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_stage_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_stage_scratch, per device ordinal

// The scratch array's device address on the current device, looked up on the
// first use on that device.  GIST_ATTN_ERR_LAUNCH if the runtime cannot give it.
int scratch_on_current_device(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GIST_ATTN_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_stage_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return GIST_ATTN_ERR_LAUNCH;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return GIST_ATTN_OK;
}

}  // namespace

extern "C" int gist_attn_fwd_noalloc(const void* q, const void* k_new, const void* v_new,
                                     const void* kv_pool, const int32_t* item_ids,
                                     const int32_t* block_table, const int32_t* pos_offset,
                                     void* out, const gist_attn_dims* dims, cudaStream_t stream) {
  // 0 for dimensions without a staged path (and for invalid ones, which the
  // call below rejects with the usual code).
  const size_t need = gist_attn_workspace_bytes(dims);
  if (need > kStaticScratchBytes) return GIST_ATTN_ERR_SCRATCH;
  void* ws = nullptr;
  if (need > 0) {
    const int rc = scratch_on_current_device(&ws);
    if (rc != GIST_ATTN_OK) return rc;
  }
  return gist_attn_fwd_ws(q, k_new, v_new, kv_pool, item_ids, block_table, pos_offset, out, ws,
                          need > 0 ? kStaticScratchBytes : 0, dims, stream);
}
