// uq_internal.h -- host-side declarations shared by the library's translation
// units (not part of the public ABI; see include/uq.h for that).
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/uq.h"

namespace uqh {

// Per-element XOR masks of the rotation's sign diagonal (0 or 0x80000000),
// passed to kernels by value so that the library keeps no device state.
struct SignMasks {
  uint32_t m[256];
};
void make_sign_masks(uint64_t seed, int d, SignMasks* out);

// Device status word of the current device (for in-kernel error records).
unsigned int* status_word();

constexpr int kMaxDevices = 64;

// Properties of the current device (cached; device = -1 when there is none).
struct DevInfo {
  int device = -1;
  int sms = 0;
  size_t smem_optin = 0;
};
const DevInfo& dev_info();

inline uq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? UQ_OK : UQ_ERR_CUDA; }

// The FP4 scale-rule constant of a cache (0 selects the default 0.156f).
inline float fp4_c(const uq_cache& c) { return c.fp4_c > 0.f ? c.fp4_c : 0.156f; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel in the stream finishes (it waits for it with
// griddepcontrol.wait before reading global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

inline int ilog2(int v) {
  int l = 0;
  while ((1 << l) < v) ++l;
  return l;
}

// TQ4 codebook tables (uq_codebook.cu), cached per head_dim: the positive
// decision thresholds tau_8..tau_14 of the 16-level codebook and the f16
// magnitudes c_0..c_7 as byte tables (lut[0..1]: high bytes of c_0..c_3,
// c_4..c_7; lut[2..3]: low bytes), the form the decode's byte permutes read.
struct TqTables {
  float tpos[7];
  uint32_t lut[4];
};
uq_status tq_tables(int d, TqTables* out);
uq_status tq_codebook_host(int d, int bits, float* mags, float* thresholds);

// Append launchers (uq_append.cu).
uq_status launch_append_fp4(const void* k, const void* v, bool in_fp32, int64_t ntok,
                            const int64_t* slots, const uq_cache& c, cudaStream_t s);  // FP4 and TQ4
uq_status launch_append_anchor(const void* k, const void* v, bool in_fp32, int64_t ntok,
                               const int64_t* slots, const uq_cache& c, cudaStream_t s);
uq_status launch_inverse_rotate(const float* x, int64_t n, int d, uint64_t seed, float* y, cudaStream_t s);
uq_status launch_test_rotate(const float* x, int64_t n, int d, uint64_t seed, float* y,
                             cudaStream_t s);
uq_status launch_test_quantize(const float* y, int64_t n, int d, uint8_t* codes, uint8_t* scales,
                               cudaStream_t s);
uq_status launch_test_cvt_e4m3(const float* x, int64_t n, uint8_t* out, cudaStream_t s);
uq_status launch_test_cvt_e2m1(const float* r, int64_t n, uint8_t* out, cudaStream_t s);
uq_status launch_test_scale_byte(const float* m, int64_t n, uint8_t* out, cudaStream_t s);
uq_status launch_calibrate(const void* x, bool in_fp32, int64_t n, int d, uint64_t seed, const float* c_list,
                           int n_c, int mode, double* sse, cudaStream_t s);

// Cascade decode: groups of consecutive sequences that share a key prefix
// (see casc_shared_keys in uq_device.cuh for the split between the kernels).
struct CascadeGroups {
  const int32_t* cu = nullptr;      // [groups + 1] first sequence of each group
  const int32_t* prefix = nullptr;  // [groups] shared keys of each group
  int32_t groups = 0;
  int32_t min_rows = 0;             // query rows a group needs to use the shared-prefix kernel
  int32_t cap = 0;                  // bound on the shared keys: min(max_pages * page_size, max_prefix_len)
};
// Partials (m, l, O) of the shared-prefix kernel, read by the decode merge.
struct PrefixPartials {
  const float* ml = nullptr;          // [items][rows][2]
  const float* o = nullptr;           // [items][rows][D]
  const int32_t* item_pre = nullptr;  // [groups + 1] work items before each group
  int32_t splits = 0;
  int32_t rows = 0;                   // query rows per work item
  int64_t max_items = 0;
};

// Decode launchers (uq_decode.cu).
struct DecodeArgs {
  const void* q;
  const uq_cache* cache;
  const int32_t* block_table;
  int32_t max_pages;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t num_q_heads;
  float sm_scale;
  float* out;
  void* ws;
  size_t ws_bytes;
  // fused append of one new token per sequence (FP4; new_slots == nullptr: none)
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  const int64_t* new_slots = nullptr;
  int new_f32 = 0;
  // cascade (FP4; casc.cu == nullptr: none): keys below each group's shared
  // prefix are skipped here and their partials px merged in
  CascadeGroups casc;
  PrefixPartials px;
};
size_t decode_workspace_bytes(int batch, int hq, int hkv, int d, int max_ctas);
int decode_max_ctas();
uq_status launch_decode(const DecodeArgs& a, cudaStream_t s);
// Injected decode timeout (test hook): arm makes the next decode launch's
// block `cta` stall (warp 0, at most budget cycles); take hands the armed
// values to that launch and disarms (cta -1: nothing armed).
void arm_decode_stall(int cta, long long budget);
void take_decode_stall(int* cta, long long* budget);
uq_status launch_query_fp8(const void* q, int64_t n, int d, uint64_t seed, uint8_t* out,
                                cudaStream_t s);

// Chunked-prefill attention (uq_prefill.cu).
struct PrefillArgs {
  const void* q;            // bf16 [T][Hq][D]
  const int32_t* cu_q;      // [B + 1]
  int32_t num_q_tokens;     // T
  const uq_cache* cache;
  const int32_t* block_table;
  int32_t max_pages;
  const int32_t* seq_lens;  // [B]
  int32_t batch;
  int32_t num_q_heads;
  float sm_scale;
  float* out;               // fp32 [T][Hq][D]
  void* ws;
  size_t ws_bytes;
};
size_t prefill_workspace_bytes(int T, int B, int hq, int hkv, int d, int max_keys);
uq_status launch_prefill(const PrefillArgs& a, cudaStream_t s);
// Shared-prefix part of a cascade decode: the query of every sequence
// (bf16 [batch][Hq][D]) against its group's first S_g keys, as partials.
size_t cascade_prefix_workspace_bytes(int batch, int groups, int hq, int hkv, int d, int max_keys);
uq_status launch_cascade_prefix(const void* q, const uq_cache* cache, const int32_t* block_table,
                                int32_t max_pages, int32_t batch, int32_t num_q_heads, const CascadeGroups& cg,
                                float sm_scale, void* ws, size_t ws_bytes, PrefixPartials* out, cudaStream_t s);

}  // namespace uqh
