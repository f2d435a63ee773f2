// uq_decode_common.cuh -- definitions shared by the two FP4 decode kernels
// (warp-level MMA in uq_decode.cu, tensor-memory MMA in uq_decode_tc.cu):
// the work split into 16-token units, the launch parameters, the partial
// layout the merge reads, and the query prologue.
#pragma once

#include <cstdint>

#include "uq_device.cuh"
#include "uq_internal.h"

namespace uqdec {

using namespace uqd;

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kHB = 8;      // query heads per block (the MMA's n)
constexpr int kChunk = 16;  // tokens per work unit (the MMA's m for QK)
// The running max M is only raised when a logit exceeds it by more than
// kSlack (log2 units); p = 2^(t - M) may then reach 2^kSlack.  p is carried as
// p * 2^kPShift, so the largest value is 2^(kSlack + kPShift) = 2^15, inside f16.
constexpr float kSlack = 8.f;
constexpr float kPShift = 7.f;
// Pair entries of the workspace hold a block index in their low kCtaBits and
// the call's epoch above them, so the merge can tell this call's entries from
// an earlier call's (the workspace is never cleared).
constexpr int kCtaBits = 12;
constexpr uint32_t kCtaMask = (1u << kCtaBits) - 1;
constexpr uint32_t kEpochMask = (1u << (32 - kCtaBits)) - 1;

enum Kind { kFP4 = 0, kFP8 = 1, kBF16 = 2, kTQ4 = 3 };
// FP4 and TQ4 share the 4-bit packed codes, the per-row side array (scale
// bytes or norm), the rotation and the two-unit main loop.
constexpr bool packed4(int kind) { return kind == kFP4 || kind == kTQ4; }

#ifndef UQ_FP4_MINB
#define UQ_FP4_MINB 3  // resident blocks per SM the FP4 decode is compiled for
#endif

template <int KIND, int D>
struct DC {
  static constexpr int KROW = packed4(KIND) ? D / 2 : (KIND == kFP8 ? D : 2 * D);  // bytes/token row
  // side bytes/token: FP4 scale bytes, TQ4 the fp32 norm
  static constexpr int SROW = KIND == kFP4 ? D / 32 : (KIND == kTQ4 ? 4 : 0);
  static constexpr int KBYTES = kChunk * KROW;
  static constexpr int SBYTES = kChunk * SROW;
  static constexpr int STAGE = 2 * KBYTES + 2 * SBYTES;
  static constexpr int NST = packed4(KIND) ? 4 : 3;  // ring depth per warp
  static constexpr int NMMA = D / 16;               // k-steps of QK, m-blocks of PV
  static constexpr int NG = D / 32;                 // 32-channel groups
  static constexpr int CPT = D / 4;                 // QK channels per thread and token
  static constexpr int VPT = D / 8;                 // PV channels per thread and token
  static constexpr size_t smem_fixed = (size_t)kWarps * NST * STAGE + (size_t)kWarps * NST * 8 +
                                       (size_t)kWarps * kHB * 2 * 4 + (size_t)kWarps * kHB * D * 4;
};

struct DecParams {
  const uint16_t* q;
  const uint8_t* kc;
  const uint8_t* ks;
  const uint8_t* vc;
  const uint8_t* vs;
  float k_scale, v_scale;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  int B, Hq, Hkv, G, nhb, ps_log2, num_pages;
  float sl2e;  // softmax scale * log2(e)
  float* ws_o;
  float* ws_ml;
  uint32_t* ws_info;  // per pair: (epoch << kCtaBits) | first block, then the same for the last block
  uint32_t epoch;     // tag of this call's pair entries (kEpochBits wide)
  int64_t* ws_units;
  unsigned int* status;
  uqh::SignMasks sign;
  uint32_t tq_lut[4];  // TQ4 codebook magnitudes as byte tables (see uqh::TqTables)
  // Fused append (FP4): new token of sequence b at physical slot new_slots[b]
  // (-1: none), rows k_new/v_new [B][Hkv][D] (bf16, or fp32 if new_f32).
  const void* k_new;
  const void* v_new;
  const int64_t* new_slots;
  int new_f32;
  int64_t num_slots;
  uint8_t* wkc;
  uint8_t* wks;
  uint8_t* wvc;
  uint8_t* wvs;
  float fp4_c;  // the scale-rule constant of the cache
  // Cascade (casc_cu == nullptr: none): the decode skips each group's shared keys.
  const int32_t* casc_cu;
  const int32_t* casc_prefix;
  int casc_groups, casc_min_rows, casc_cap;
  // Injected timeout (test hook; stall_cta < 0: none): warp 0 of block
  // stall_cta also waits, at its first unit, on a barrier that nothing
  // arrives at, for at most stall_budget cycles, and so takes the timeout path.
  int stall_cta;
  long long stall_budget;
};

// Contiguous range [lo, hi) of the U units that block c of C handles.
__device__ __forceinline__ void block_range(int64_t c, int64_t U, int64_t C, int64_t& lo, int64_t& hi) {
  lo = c * U / C;
  hi = (c + 1) * U / C;
}

__device__ __forceinline__ float pow2i(int e) {  // 2^e for e in [-149, 127], 0 below
  if (e >= -126) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  if (e >= -149) return __uint_as_float(1u << (e + 149));
  return 0.f;
}

// 2^(byte-127) as fp32 for the byte at bit offset 8*g of w: the byte becomes
// the exponent field.  Byte 0 gives +0 instead of 2^-127 (a group that small
// contributes nothing representable); byte 0xFF gives +Inf, so a non-finite
// group poisons the logit.
template <int G>
__device__ __forceinline__ float scale_of(uint32_t w) {
  return G == 3 ? __uint_as_float((w >> 1) & 0x7F800000u)
                : __uint_as_float((w << (23 - 8 * G)) & 0x7F800000u);
}

// Non-zero if any byte of w is 0xFF (a non-finite group).
__device__ __forceinline__ uint32_t has_ff(uint32_t w) {
  return ((w & 0x7F7F7F7Fu) + 0x01010101u) & w & 0x80808080u;
}

// Keys of sequence b attended by the shared-prefix kernel of a cascade decode
// (a multiple of 16; 0 without cascade).
template <typename P>
__device__ __forceinline__ int casc_skip(const P& p, int b) {
  if (p.casc_cu == nullptr) return 0;
  const int g = casc_group(p.casc_cu, p.casc_groups, b);
  if (g < 0) return 0;
  return casc_shared_keys(p.casc_cu[g + 1] - p.casc_cu[g], p.G, p.casc_prefix[g], p.casc_min_rows, p.casc_cap);
}

__device__ __forceinline__ int clamp_len(const DecParams& p, int b) {
  const int cap = p.max_pages << p.ps_log2;
  int L = p.seq_lens[b];
  if (L < 0 || L > cap) {
    record_error(p.status, kErrBounds);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

// R1 rotation of one row of D values spread over the 4 threads of a quad:
// thread c ends with rotated channels [c*D/4, (c+1)*D/4) in fp32.  The same
// fp32 butterfly as the append path (strides below D/4 inside a thread, the
// last two across the quad, ascending), then the 1/sqrt(D) factor.  Every
// lane of the warp must call it (the cross-quad steps are warp shuffles).
template <int D, bool F32>
__device__ __forceinline__ void rotate_quad(const void* row, bool valid, int c, const uqh::SignMasks& sign,
                                            float (&x)[D / 4]) {
  constexpr int CPT = D / 4;
  if (F32) {
#pragma unroll
    for (int e = 0; e < CPT; ++e) {
      const uint32_t w = valid ? reinterpret_cast<const uint32_t*>(row)[c * CPT + e] : 0u;
      x[e] = __uint_as_float(w ^ sign.m[c * CPT + e]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < CPT; e += 2) {
      const uint32_t w = valid ? *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(row) + c * CPT + e) : 0u;
      x[e] = __uint_as_float((w << 16) ^ sign.m[c * CPT + e]);
      x[e + 1] = __uint_as_float((w & 0xFFFF0000u) ^ sign.m[c * CPT + e + 1]);
    }
  }
  fwht_regs<CPT>(x);
#pragma unroll
  for (int k = 1; k <= 2; k <<= 1) {
    const bool upper = (c & k) != 0;
#pragma unroll
    for (int e = 0; e < CPT; ++e) {
      const float o = __shfl_xor_sync(kFull, x[e], k);
      x[e] = upper ? (o - x[e]) : (x[e] + o);
    }
  }
  const float s = inv_sqrt_d<D>();
#pragma unroll
  for (int e = 0; e < CPT; e += 2) mul2(x[e], x[e + 1], s);
}

// The rotated E4M3 query of one head, channels [c*D/4, (c+1)*D/4), packed 4
// bytes per word, E4M3 round to nearest even, saturating.
template <int D>
__device__ __forceinline__ void rotated_query_bytes(const uint16_t* qrow, bool valid, int c,
                                                    const uqh::SignMasks& sign, uint32_t (&out)[D / 16]) {
  float x[D / 4];
  rotate_quad<D, false>(qrow, valid, c, sign, x);
#pragma unroll
  for (int m = 0; m < D / 16; ++m)
    out[m] = cvt_e4m3x2(x[4 * m], x[4 * m + 1]) | (cvt_e4m3x2(x[4 * m + 2], x[4 * m + 3]) << 16);
}

// R2 + R3 on the rotated channels a quad thread holds (32 for D = 128, one
// group; 16 for D = 64, half a group shared with the neighbouring thread):
// the group's UE8M0 byte and the E2M1 codes of this thread's channels, with
// the same arithmetic as the append path.  All lanes must call it.
template <int D>
__device__ __forceinline__ void quantize_quad(float (&x)[D / 4], uint32_t (&codes)[D / 32], uint32_t& byte,
                                              float c) {
  constexpr int CPT = D / 4;
  float mx = max_abs_nan(x[0], x[1]);
#pragma unroll
  for (int i = 2; i < CPT; ++i) mx = max_abs_nan(mx, x[i]);
  if (CPT < 32) mx = max_abs_nan(mx, __shfl_xor_sync(kFull, mx, 1));
  byte = scale_byte(fabsf(mx), c);
  const float inv = inv_scale(byte == 0xFFu ? 127u : byte);
#pragma unroll
  for (int i = 0; i < CPT; i += 2) mul2(x[i], x[i + 1], inv);
#pragma unroll
  for (int w = 0; w < CPT / 8; ++w) {
    const float* e = &x[8 * w];
    const uint32_t word = cvt_e2m1x2(e[0], e[1]) | (cvt_e2m1x2(e[2], e[3]) << 8) |
                          (cvt_e2m1x2(e[4], e[5]) << 16) | (cvt_e2m1x2(e[6], e[7]) << 24);
    codes[w] = byte == 0xFFu ? 0u : word;
  }
}

// The tensor-memory FP4 decode (uq_decode_tc.cu), head_dim 128, page size >= 16:
// same parameters, work split and partials as decode_kernel, one CTA per SM.
bool decode_tc_enabled();
size_t decode_tc_smem(int batch);
uq_status launch_decode_tc(const DecParams& p, int grid, cudaStream_t s);

}  // namespace uqdec
