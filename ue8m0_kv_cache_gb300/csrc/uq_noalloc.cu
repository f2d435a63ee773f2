// uq_noalloc.cu -- a decode-attention entry point for callers that cannot
// allocate device memory.
//
// uq_decode_attention needs a caller-provided workspace for its split-K
// partials.  Some callers have no way to provide one: their device memory is
// owned by another allocator (a framework's caching allocator or a fixed
// arena) that they may not draw from on the decode path, and they may not call
// cudaMalloc themselves either.  For them, uq_decode_attention_noalloc uses a
// fixed scratch array that lives in the library's own device image instead.
//
// The scratch is a file-scope __device__ array of kScratchBytes.  Every GPU on
// which the library is loaded holds it until the process exits.  In host code
// the array's name does not denote a device address, so the address is looked
// up with cudaGetSymbolAddress (with the device current) and passed to the
// kernels.  The address is kept per device together with the identity of the
// context it was read in, and read again when the device's current context
// is a different one (after cudaDeviceReset, for instance).
#include <cuda.h>

#include <mutex>

#include "uq_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

}  // namespace

static __device__ __align__(256) unsigned char uq_noalloc_scratch[kScratchBytes];

namespace {

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];
unsigned long long g_scratch_ctx[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (the driver numbers every
// context it creates), or 0 when it cannot be read.  The two driver entry
// points are fetched through the runtime once; the library links no driver
// library of its own.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current device's current
// context.  The first call on a device (and the first after the context was
// replaced) looks it up, which may load the library's device code.
uq_status scratch_for_current_device(void** ptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return UQ_ERR_CUDA;
  unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, uq_noalloc_scratch) != cudaSuccess || p == nullptr) return UQ_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx != 0 ? ctx : current_context_id();  // the lookup may have made the context current
  }
  *ptr = g_scratch_ptr[dev];
  return UQ_OK;
}

}  // namespace

extern "C" uq_status uq_decode_attention_noalloc(const void* q, const uq_cache* cache,
                                                 const int32_t* block_table, int32_t max_pages_per_seq,
                                                 const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                                 float sm_scale, float* out, cudaStream_t stream) {
  if (!cache || cache->num_kv_heads <= 0 || num_q_heads <= 0 || batch < 0 || cache->head_dim <= 0)
    return UQ_ERR_INVALID_ARG;
  if (num_q_heads % cache->num_kv_heads != 0) return UQ_ERR_INVALID_ARG;
  if (batch == 0) return UQ_OK;
  if (batch > 4096) return UQ_ERR_UNSUPPORTED;  // as uq_decode_attention; checked before any size arithmetic
  // The smallest workspace the decode accepts: one block plus one partial per
  // (sequence, kv head, head block).  Shapes that need more than the static
  // scratch holds are rejected here, before anything is enqueued.
  const size_t need = uqh::decode_workspace_bytes(batch, num_q_heads, cache->num_kv_heads, cache->head_dim, 1);
  if (need > kScratchBytes) return UQ_ERR_WORKSPACE;
  void* ws = nullptr;
  const uq_status st = scratch_for_current_device(&ws);
  if (st != UQ_OK) return st;
  return uq_decode_attention(q, cache, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale,
                             out, ws, kScratchBytes, stream);
}
