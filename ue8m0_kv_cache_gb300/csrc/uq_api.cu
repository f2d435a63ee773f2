// uq_api.cu -- the extern "C" entry points of libuq.so (declared in
// include/uq.h): argument validation, dispatch to the kernels, the device
// status word, and the host-side sign generator of the rotation.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "uq_internal.h"

// One status word per device: kernels record the first bounds violation or
// wait timeout here instead of faulting or hanging.
__device__ unsigned int uq_device_status_word;

namespace uqh {

namespace {

// splitmix64 (Steele, Lea, Flood 2014): output i of the stream seeded with
// `seed` is the finaliser applied to seed + (i + 1) * 0x9E3779B97F4A7C15.
uint64_t splitmix64_at(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

std::mutex g_mu;
unsigned int* g_status[kMaxDevices];
DevInfo g_info[kMaxDevices];

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

}  // namespace

void make_sign_masks(uint64_t seed, int d, SignMasks* out) {
  std::memset(out, 0, sizeof(*out));
  for (int i = 0; i < d && i < 256; ++i) out->m[i] = (splitmix64_at(seed, i) >> 63) ? 0x80000000u : 0u;
}

unsigned int* status_word() {
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, uq_device_status_word) != cudaSuccess) return nullptr;
    g_status[d] = static_cast<unsigned int*>(p);
  }
  return g_status[d];
}

const DevInfo& dev_info() {
  static DevInfo none;
  const int d = current_device();
  if (d < 0) return none;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& di = g_info[d];
  if (di.device != d) {
    int sms = 0, optin = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    di.sms = sms;
    di.smem_optin = static_cast<size_t>(optin);
    di.device = d;
  }
  return di;
}

}  // namespace uqh

namespace {

using uqh::aligned16;

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

// Shape and pointer checks common to append and decode.
uq_status check_cache(const uq_cache* c) {
  if (!c) return UQ_ERR_INVALID_ARG;
  if (c->dtype < UQ_FP4_UE8M0 || c->dtype > UQ_TQ4) return UQ_ERR_INVALID_ARG;
  if (c->num_pages <= 0 || c->num_kv_heads <= 0 || c->page_size <= 0 || c->head_dim <= 0)
    return UQ_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return UQ_ERR_UNSUPPORTED;
  if (c->head_dim == 256 && c->dtype == UQ_TQ4) return UQ_ERR_UNSUPPORTED;
  if (!is_pow2(c->page_size) || c->page_size < 16 || c->page_size > 256) return UQ_ERR_UNSUPPORTED;
  if ((int64_t)c->num_pages * c->num_kv_heads * c->page_size >= (int64_t(1) << 40)) return UQ_ERR_UNSUPPORTED;
  if (!c->k_codes || !c->v_codes) return UQ_ERR_INVALID_ARG;
  const bool packed = c->dtype == UQ_FP4_UE8M0 || c->dtype == UQ_TQ4;  // codes + per-row side array
  if (packed && (!c->k_scales || !c->v_scales)) return UQ_ERR_INVALID_ARG;
  if (!aligned16(c->k_codes) || !aligned16(c->v_codes)) return UQ_ERR_ALIGNMENT;
  if (packed && (!aligned16(c->k_scales) || !aligned16(c->v_scales))) return UQ_ERR_ALIGNMENT;
  if (c->dtype == UQ_FP8_E4M3 && !(c->k_scale > 0.f && c->v_scale > 0.f)) return UQ_ERR_INVALID_ARG;
  if (!(c->fp4_c >= 0.f && c->fp4_c <= 3.4e38f)) return UQ_ERR_INVALID_ARG;
  return UQ_OK;
}

uq_status decode_common(const void* q, const uq_cache* cache, const int32_t* block_table, int32_t max_pages,
                        const int32_t* seq_lens, int32_t batch, int32_t hq, float sm_scale, float* out,
                        void* ws, size_t ws_bytes, cudaStream_t stream, int want_dtype,
                        const void* k_new = nullptr, const void* v_new = nullptr,
                        const int64_t* new_slots = nullptr, int new_f32 = 0) {
  uq_status st = check_cache(cache);
  if (st != UQ_OK) return st;
  if (want_dtype >= 0 && cache->dtype != want_dtype) return UQ_ERR_INVALID_ARG;
  if (batch < 0 || hq <= 0 || max_pages < 0) return UQ_ERR_INVALID_ARG;
  if (hq % cache->num_kv_heads != 0) return UQ_ERR_INVALID_ARG;
  if (batch == 0) return UQ_OK;
  if (batch > 4096) return UQ_ERR_UNSUPPORTED;
  if (!q || !block_table || !seq_lens || !out || !ws) return UQ_ERR_INVALID_ARG;
  if (max_pages < 1) return UQ_ERR_INVALID_ARG;
  if ((int64_t)max_pages * cache->page_size >= (int64_t(1) << 31)) return UQ_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(out) || !aligned16(ws)) return UQ_ERR_ALIGNMENT;
  uqh::DecodeArgs a{q, cache, block_table, max_pages, seq_lens, batch, hq, sm_scale, out, ws, ws_bytes};
  a.k_new = k_new;
  a.v_new = v_new;
  a.new_slots = new_slots;
  a.new_f32 = new_f32;
  return uqh::launch_decode(a, stream);
}

}  // namespace

extern "C" {

size_t uq_cache_bytes(const uq_cache* c, int32_t which) {
  if (!c || c->num_pages <= 0 || c->num_kv_heads <= 0 || c->page_size <= 0 || c->head_dim <= 0) return 0;
  const size_t rows = (size_t)c->num_pages * c->num_kv_heads * c->page_size;
  switch (c->dtype) {
    case UQ_FP4_UE8M0:
      if (which == 0 || which == 2) return rows * (c->head_dim / 2);
      if (which == 1 || which == 3) return rows * (c->head_dim / 32);
      return 0;
    case UQ_FP8_E4M3:
      return (which == 0 || which == 2) ? rows * c->head_dim : 0;
    case UQ_BF16:
      return (which == 0 || which == 2) ? rows * c->head_dim * 2 : 0;
    case UQ_TQ4:
      if (which == 0 || which == 2) return rows * (c->head_dim / 2);
      if (which == 1 || which == 3) return rows * sizeof(float);
      return 0;
    default:
      return 0;
  }
}

uq_status uq_quantize_append(const void* k, const void* v, int32_t in_dtype, int64_t num_tokens,
                             const int32_t* block_table, int32_t max_pages_per_seq, const int64_t* slot_mapping,
                             const uq_cache* cache, cudaStream_t stream) {
  (void)block_table;
  (void)max_pages_per_seq;
  uq_status st = check_cache(cache);
  if (st != UQ_OK) return st;
  if (in_dtype != UQ_IN_BF16 && in_dtype != UQ_IN_FP32) return UQ_ERR_INVALID_ARG;
  if (num_tokens < 0) return UQ_ERR_INVALID_ARG;
  if (num_tokens == 0) return UQ_OK;
  if (!k || !v || !slot_mapping) return UQ_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v)) return UQ_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0) return UQ_ERR_ALIGNMENT;
  const bool f32 = in_dtype == UQ_IN_FP32;
  if (cache->dtype == UQ_FP4_UE8M0 || cache->dtype == UQ_TQ4)
    return uqh::launch_append_fp4(k, v, f32, num_tokens, slot_mapping, *cache, stream);
  return uqh::launch_append_anchor(k, v, f32, num_tokens, slot_mapping, *cache, stream);
}

size_t uq_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_q_heads % num_kv_heads)
    return 0;
  const int max_ctas = uqh::decode_max_ctas();
  return uqh::decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_ctas > 0 ? max_ctas : 1);
}

uq_status uq_decode_attention(const void* q, const uq_cache* cache, const int32_t* block_table,
                              int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                              int32_t num_q_heads, float sm_scale, float* out, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  return decode_common(q, cache, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale, out,
                       workspace, workspace_bytes, stream, -1);
}

uq_status uq_decode_attention_append(const void* q, const void* k_new, const void* v_new, int32_t in_dtype,
                                     const int64_t* new_slots, const uq_cache* cache, const int32_t* block_table,
                                     int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                                     int32_t num_q_heads, float sm_scale, float* out, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream) {
  if (!cache) return UQ_ERR_INVALID_ARG;
  if (cache->dtype != UQ_FP4_UE8M0 || cache->head_dim == 256) return UQ_ERR_UNSUPPORTED;
  if (in_dtype != UQ_IN_BF16 && in_dtype != UQ_IN_FP32) return UQ_ERR_INVALID_ARG;
  if (batch > 0 && (!k_new || !v_new || !new_slots)) return UQ_ERR_INVALID_ARG;
  if (batch > 0 && (!aligned16(k_new) || !aligned16(v_new))) return UQ_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(new_slots) & 7u) != 0) return UQ_ERR_ALIGNMENT;
  return decode_common(q, cache, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale, out,
                       workspace, workspace_bytes, stream, UQ_FP4_UE8M0, k_new, v_new, new_slots,
                       in_dtype == UQ_IN_FP32 ? 1 : 0);
}

uq_status uq_decode_attention_fp8(const void* q, const uq_cache* cache, const int32_t* block_table,
                                  int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                                  int32_t num_q_heads, float sm_scale, float* out, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
  return decode_common(q, cache, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale, out,
                       workspace, workspace_bytes, stream, UQ_FP8_E4M3);
}

uq_status uq_decode_attention_bf16(const void* q, const uq_cache* cache, const int32_t* block_table,
                                   int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                                   int32_t num_q_heads, float sm_scale, float* out, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream) {
  return decode_common(q, cache, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale, out,
                       workspace, workspace_bytes, stream, UQ_BF16);
}

uq_status uq_decode_attention_tq4(const void* q, const uq_cache* cache, const int32_t* block_table,
                                  int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                                  int32_t num_q_heads, float sm_scale, float* out, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
  return decode_common(q, cache, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale, out,
                       workspace, workspace_bytes, stream, UQ_TQ4);
}

size_t uq_prefill_workspace_bytes(int32_t num_q_tokens, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_keys) {
  if (num_q_tokens < 0 || batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
      (head_dim != 64 && head_dim != 128) || max_keys <= 0)
    return 0;
  return uqh::prefill_workspace_bytes(num_q_tokens, batch, num_q_heads, num_kv_heads, head_dim, max_keys);
}

uq_status uq_prefill_attention(const void* q, const int32_t* cu_q, int32_t num_q_tokens, const uq_cache* cache,
                               const int32_t* block_table, int32_t max_pages_per_seq, const int32_t* seq_lens,
                               int32_t batch, int32_t num_q_heads, float sm_scale, float* out, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  uq_status st = check_cache(cache);
  if (st != UQ_OK) return st;
  if (cache->dtype != UQ_FP4_UE8M0 || cache->head_dim == 256) return UQ_ERR_UNSUPPORTED;
  if (batch < 0 || num_q_tokens < 0 || num_q_heads <= 0 || max_pages_per_seq < 1) return UQ_ERR_INVALID_ARG;
  if (num_q_heads % cache->num_kv_heads != 0) return UQ_ERR_INVALID_ARG;
  if (batch == 0 || num_q_tokens == 0) return UQ_OK;
  if (batch > 65536) return UQ_ERR_UNSUPPORTED;
  if ((int64_t)max_pages_per_seq * cache->page_size >= (int64_t(1) << 31)) return UQ_ERR_UNSUPPORTED;
  if (!q || !cu_q || !block_table || !seq_lens || !out || !workspace) return UQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace)) return UQ_ERR_ALIGNMENT;
  uqh::PrefillArgs a{q, cu_q, num_q_tokens, cache, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads,
                     sm_scale, out, workspace, workspace_bytes};
  return uqh::launch_prefill(a, stream);
}

size_t uq_cascade_workspace_bytes(int32_t batch, int32_t num_groups, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_prefix_len) {
  const size_t dec = uq_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim);
  if (dec == 0 || num_groups < 0 || max_prefix_len < 0 || (head_dim != 64 && head_dim != 128)) return 0;
  const size_t pre = num_groups > 0 ? uqh::cascade_prefix_workspace_bytes(batch, num_groups, num_q_heads,
                                                                         num_kv_heads, head_dim, max_prefix_len)
                                    : 0;
  return ((dec + 255) & ~size_t(255)) + pre;
}

uq_status uq_cascade_decode_attention(const void* q, const uq_cache* cache, const int32_t* block_table,
                                      int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                                      int32_t num_q_heads, const int32_t* cu_seqs, const int32_t* prefix_lens,
                                      int32_t num_groups, int32_t max_prefix_len, int32_t min_rows, float sm_scale,
                                      float* out, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  uq_status st = check_cache(cache);
  if (st != UQ_OK) return st;
  if (cache->dtype != UQ_FP4_UE8M0) return UQ_ERR_UNSUPPORTED;
  if (cache->head_dim != 64 && cache->head_dim != 128) return UQ_ERR_UNSUPPORTED;
  if (num_groups < 0 || max_prefix_len < 0 || min_rows < 0) return UQ_ERR_INVALID_ARG;
  if (num_groups > 0 && (!cu_seqs || !prefix_lens)) return UQ_ERR_INVALID_ARG;
  if (batch <= 0 || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0)
    return decode_common(q, cache, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale, out,
                         workspace, workspace_bytes, stream, UQ_FP4_UE8M0);
  const size_t dec = uq_decode_workspace_bytes(batch, num_q_heads, cache->num_kv_heads, cache->head_dim);
  const size_t dec_al = (dec + 255) & ~size_t(255);
  const int G = num_q_heads / cache->num_kv_heads;
  const int64_t cap = std::min<int64_t>(static_cast<int64_t>(max_pages_per_seq) * cache->page_size, max_prefix_len);
  // No group can reach min_rows, or nothing to share: a plain decode.
  if (num_groups == 0 || cap < 16 || static_cast<int64_t>(batch) * G < min_rows)
    return decode_common(q, cache, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale, out,
                         workspace, workspace_bytes, stream, UQ_FP4_UE8M0);
  if (!q || !block_table || !seq_lens || !out || !workspace) return UQ_ERR_INVALID_ARG;
  if (max_pages_per_seq < 1 || batch > 4096) return UQ_ERR_INVALID_ARG;
  if ((int64_t)max_pages_per_seq * cache->page_size >= (int64_t(1) << 31)) return UQ_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace)) return UQ_ERR_ALIGNMENT;
  if (workspace_bytes < dec_al) return UQ_ERR_WORKSPACE;
  uqh::CascadeGroups cg;
  cg.cu = cu_seqs;
  cg.prefix = prefix_lens;
  cg.groups = num_groups;
  cg.min_rows = min_rows;
  cg.cap = static_cast<int32_t>(cap);
  uqh::PrefixPartials px;
  st = uqh::launch_cascade_prefix(q, cache, block_table, max_pages_per_seq, batch, num_q_heads, cg, sm_scale,
                                  static_cast<uint8_t*>(workspace) + dec_al, workspace_bytes - dec_al, &px, stream);
  if (st != UQ_OK) return st;
  uqh::DecodeArgs a{q, cache, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale, out,
                    workspace, dec};
  a.casc = cg;
  a.px = px;
  return uqh::launch_decode(a, stream);
}

uq_status uq_calibrate_c(const void* x, int32_t in_dtype, int64_t n_vec, int32_t head_dim, uint64_t rot_seed,
                         const float* c_list, int32_t n_c, int32_t mode, double* sse, cudaStream_t stream) {
  if (in_dtype != UQ_IN_BF16 && in_dtype != UQ_IN_FP32) return UQ_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return UQ_ERR_UNSUPPORTED;
  if (n_vec < 0 || n_c < 1 || n_c > 64 || (mode != 0 && mode != -1) || !c_list || !sse) return UQ_ERR_INVALID_ARG;
  if (n_vec > 0 && !x) return UQ_ERR_INVALID_ARG;
  for (int i = 0; i < n_c; ++i)
    if (!(c_list[i] > 0.f && c_list[i] <= 3.4e38f)) return UQ_ERR_INVALID_ARG;
  if (n_vec > 0 && !aligned16(x)) return UQ_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(sse) & 7u) != 0) return UQ_ERR_ALIGNMENT;
  return uqh::launch_calibrate(x, in_dtype == UQ_IN_FP32, n_vec, head_dim, rot_seed, c_list, n_c, mode, sse, stream);
}

uq_status uq_check_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return UQ_ERR_CUDA;
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, uq_device_status_word, sizeof(v)) != cudaSuccess) return UQ_ERR_CUDA;
  if (v != 0 && cudaMemcpyToSymbol(uq_device_status_word, &zero, sizeof(zero)) != cudaSuccess) return UQ_ERR_CUDA;
  if (v == UQ_ERR_DEVICE_TIMEOUT || v == UQ_ERR_DEVICE_BOUNDS) return static_cast<uq_status>(v);
  return v == 0 ? UQ_OK : UQ_ERR_CUDA;
}

const char* uq_status_string(uq_status s) {
  switch (s) {
    case UQ_OK: return "UQ_OK";
    case UQ_ERR_INVALID_ARG: return "UQ_ERR_INVALID_ARG";
    case UQ_ERR_UNSUPPORTED: return "UQ_ERR_UNSUPPORTED";
    case UQ_ERR_ALIGNMENT: return "UQ_ERR_ALIGNMENT";
    case UQ_ERR_WORKSPACE: return "UQ_ERR_WORKSPACE";
    case UQ_ERR_CUDA: return "UQ_ERR_CUDA";
    case UQ_ERR_DEVICE_TIMEOUT: return "UQ_ERR_DEVICE_TIMEOUT";
    case UQ_ERR_DEVICE_BOUNDS: return "UQ_ERR_DEVICE_BOUNDS";
    default: return "UQ_ERR_UNKNOWN";
  }
}

void uq_rotation_signs(uint64_t seed, int32_t d, int8_t* host_out) {
  if (!host_out || d <= 0) return;
  for (int32_t i = 0; i < d; ++i) host_out[i] = (uqh::splitmix64_at(seed, i) >> 63) ? -1 : 1;
}

uq_status uq_test_rotate(const float* x, int64_t n_vec, int32_t d, uint64_t seed, int32_t inverse, float* y,
                         cudaStream_t stream) {
  if ((d != 64 && d != 128 && d != 256) || n_vec < 0) return UQ_ERR_UNSUPPORTED;
  if (inverse != 0 && inverse != 1) return UQ_ERR_INVALID_ARG;
  if (n_vec == 0) return UQ_OK;
  if (!x || !y) return UQ_ERR_INVALID_ARG;
  if (inverse) return uqh::launch_inverse_rotate(x, n_vec, d, seed, y, stream);
  return uqh::launch_test_rotate(x, n_vec, d, seed, y, stream);
}

uq_status uq_test_quantize_rotated(const float* y, int64_t n_vec, int32_t d, uint8_t* codes, uint8_t* scales,
                                   cudaStream_t stream) {
  if ((d != 64 && d != 128 && d != 256) || n_vec < 0) return UQ_ERR_UNSUPPORTED;
  if (n_vec == 0) return UQ_OK;
  if (!y || !codes || !scales) return UQ_ERR_INVALID_ARG;
  if (!aligned16(codes)) return UQ_ERR_ALIGNMENT;
  return uqh::launch_test_quantize(y, n_vec, d, codes, scales, stream);
}

uq_status uq_test_query_fp8(const void* q, int64_t n_vec, int32_t d, uint64_t seed, uint8_t* out,
                            cudaStream_t stream) {
  if ((d != 64 && d != 128 && d != 256) || n_vec < 0) return UQ_ERR_UNSUPPORTED;
  if (n_vec == 0) return UQ_OK;
  if (!q || !out) return UQ_ERR_INVALID_ARG;
  if (!aligned16(q)) return UQ_ERR_ALIGNMENT;
  return uqh::launch_query_fp8(q, n_vec, d, seed, out, stream);
}

uq_status uq_test_cvt_e2m1(const float* r, int64_t n, uint8_t* codes, cudaStream_t stream) {
  if (n < 0 || (n & 1)) return UQ_ERR_INVALID_ARG;
  if (n == 0) return UQ_OK;
  if (!r || !codes) return UQ_ERR_INVALID_ARG;
  return uqh::launch_test_cvt_e2m1(r, n, codes, stream);
}

uq_status uq_test_scale_byte(const float* m, int64_t n, uint8_t* bytes, cudaStream_t stream) {
  if (n < 0) return UQ_ERR_INVALID_ARG;
  if (n == 0) return UQ_OK;
  if (!m || !bytes) return UQ_ERR_INVALID_ARG;
  return uqh::launch_test_scale_byte(m, n, bytes, stream);
}

uq_status uq_test_cvt_e4m3(const float* x, int64_t n, uint8_t* out, cudaStream_t stream) {
  if (n < 0 || (n & 1)) return UQ_ERR_INVALID_ARG;
  if (n == 0) return UQ_OK;
  if (!x || !out) return UQ_ERR_INVALID_ARG;
  return uqh::launch_test_cvt_e4m3(x, n, out, stream);
}

uq_status uq_test_arm_decode_timeout(int32_t cta, int64_t budget_cycles) {
  if (cta < 0 || budget_cycles < 0) return UQ_ERR_INVALID_ARG;
  uqh::arm_decode_stall(cta, static_cast<long long>(budget_cycles));
  return UQ_OK;
}

}  // extern "C"
