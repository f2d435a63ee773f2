// uq_append.cu -- quantize-append kernels.
//
// FP4 path ("UltraQuant" review, manon006.tistory.com/395, §3.1): each K and
// V row of head_dim values is rotated by the randomised Walsh-Hadamard
// transform, split into 32-channel groups, given a UE8M0 scale byte from the
// group absmax times c = 0.156 (§3.3), and coded as E2M1 nibbles, 17 bytes
// per 32 elements, written into its paged slot.
//
// TQ4 path (the TurboQuant Q_mse codebook variant, "TurboQuant 완전 정리",
// juhoplayground.github.io, "Lloyd-Max 스칼라 양자화 (Q_mse)"): the same rotation,
// then the row's L2 norm and one 4-bit index of the nearest Lloyd-Max
// centroid per coordinate of the unit vector; same page layout, the norm in
// place of the scale bytes.
//
// GB300 mapping: one thread owns one row (128 values live in registers, so the
// whole butterfly needs no shuffles or shared-memory exchange).  Tiles of 64
// token-head rows of K and of V are brought into shared memory by 2-D TMA
// copies with the 128-byte swizzle, which makes the per-thread row reads
// bank-conflict free; a two-stage ring overlaps the next tile's copy with the
// current tile's arithmetic.  The grid is persistent (a multiple of the SM
// count).  The kernel is HBM-bound in principle (512 B read and 136 B written
// per token-head for bf16 input).
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>

#include "uq_device.cuh"
#include "uq_internal.h"

namespace {

using namespace uqd;

constexpr int kRows = 64;             // token-head rows per tile
constexpr int kAppendStages = 2;      // tiles in the ring of the tiled kernel (all but one in flight)
constexpr int64_t kSmallAppendRows = 1024;  // token-head rows up to which the direct-load kernel is used
constexpr int kAppendThreads = 2 * kRows;  // one thread per K row and one per V row

struct AppendParams {
  const int64_t* slots;
  int64_t ntok;
  int hkv;
  int ps_log2;
  int64_t num_slots;
  uint8_t* kc;
  uint8_t* ks;
  uint8_t* vc;
  uint8_t* vs;
  unsigned int* status;
  uqh::SignMasks sign;
  float tq_tpos[7];  // TQ4: positive decision thresholds tau_8..tau_14
  float c;           // FP4: the constant of the scale rule
};

// Rotation of a register-resident row whose signs were already applied.
template <int D>
__device__ __forceinline__ void rotate_regs(float (&u)[D]) {
  fwht_regs<D>(u);
  const float c = inv_sqrt_d<D>();
#pragma unroll
  for (int i = 0; i < D; i += 2) mul2(u[i], u[i + 1], c);
}

// Quantiser stage on a rotated row: codes[w] holds bytes 4w..4w+3 of the
// row's D/2 code bytes, `scales` the D/32 scale bytes (little-endian).
template <int D>
__device__ __forceinline__ void quantize_regs(float (&y)[D], uint32_t (&codes)[D / 8],
                                              uint64_t& scales, float c = kFp4C) {
  scales = 0;
#pragma unroll
  for (int g = 0; g < D / 32; ++g) {
    float mx = max_abs_nan(y[32 * g], y[32 * g + 1]);
#pragma unroll
    for (int i = 2; i < 32; ++i) mx = max_abs_nan(mx, y[32 * g + i]);
    const uint32_t byte = scale_byte(fabsf(mx), c);
    const float inv = inv_scale(byte == 0xFFu ? 127u : byte);
#pragma unroll
    for (int i = 0; i < 32; i += 2) mul2(y[32 * g + i], y[32 * g + i + 1], inv);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float* e = &y[32 * g + 8 * w];
      uint32_t word = cvt_e2m1x2(e[0], e[1]) | (cvt_e2m1x2(e[2], e[3]) << 8) |
                      (cvt_e2m1x2(e[4], e[5]) << 16) | (cvt_e2m1x2(e[6], e[7]) << 24);
      codes[4 * g + w] = byte == 0xFFu ? 0u : word;
    }
    scales |= static_cast<uint64_t>(byte) << (8 * g);
  }
}

// TQ4 quantiser on a rotated row (codes as quantize_regs; `norm_bits` the fp32
// norm).  The norm is fl32(sqrt(S)) with S the fp32 sum of the squares over a
// balanced binary tree of adjacent elements (left half + right half,
// recursively), evaluated here as a binary counter so that only log2(D)
// partial sums are live.  With t_k = fl32(n * tau_k), a coordinate y >= 0 gets
// the magnitude rank #{k : y >= t_k} and y < 0 gets 8 | #{k : |y| > t_k}; on
// the bit patterns of non-negative floats (ordered like the values) both
// counts are #{k : key >= bits(t_k)} with key = bits(|y|) - (y < 0), found by
// a three-step binary search over the sorted thresholds.
template <int D>
__device__ __forceinline__ void quantize_tq_regs(const float (&y)[D], uint32_t (&codes)[D / 8],
                                                 uint32_t& norm_bits, const float (&tpos)[7]) {
  float partial[8];
  float S = 0.f;
#pragma unroll
  for (int i = 0; i < D; ++i) {
    float v = __fmul_rn(y[i], y[i]);
#pragma unroll
    for (int lvl = 0; lvl < 8; ++lvl) {
      if (((i + 1) >> lvl) & 1) {
        partial[lvl] = v;
        break;
      }
      v = __fadd_rn(partial[lvl], v);
    }
    if (i == D - 1) S = v;
  }
  const float n = __fsqrt_rn(S);
  if (!(n <= 3.402823466e38f)) {  // NaN or Inf
    norm_bits = 0x7FC00000u;
#pragma unroll
    for (int w = 0; w < D / 8; ++w) codes[w] = 0u;
    return;
  }
  norm_bits = __float_as_uint(n);
  uint32_t tb[7];
#pragma unroll
  for (int k = 0; k < 7; ++k) tb[k] = __float_as_uint(__fmul_rn(n, tpos[k]));
#pragma unroll
  for (int w = 0; w < D / 8; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x = y[8 * w + e];
      const uint32_t neg = x < 0.f ? 1u : 0u;
      const uint32_t key = (__float_as_uint(x) & 0x7FFFFFFFu) - neg;
      uint32_t m = key >= tb[3] ? 4u : 0u;
      m += key >= (m ? tb[5] : tb[1]) ? 2u : 0u;
      const uint32_t t1 = (m & 4u) ? ((m & 2u) ? tb[6] : tb[4]) : ((m & 2u) ? tb[2] : tb[0]);
      m += key >= t1 ? 1u : 0u;
      word |= ((neg << 3) | m) << (4 * e);
    }
    codes[w] = word;
  }
}

// Store one quantised row: codes[4g + w] is word w (bytes 4w..4w+3) of group
// g in natural order.  K rows (KPERM) are stored group-interleaved by words --
// word w of group g at word position (D/32)*w + g -- so that the decode can
// fetch one word of every group with a single aligned load; V rows keep the
// natural order.
template <int D, bool KPERM, bool TQ = false>
__device__ __forceinline__ void store_row(uint8_t* codes_base, uint8_t* scales_base, int64_t row,
                                          const uint32_t (&codes)[D / 8], uint64_t scales) {
  constexpr int NG = D / 32;
  uint32_t out[D / 8];
#pragma unroll
  for (int g = 0; g < NG; ++g)
#pragma unroll
    for (int w = 0; w < 4; ++w) out[KPERM ? NG * w + g : 4 * g + w] = codes[4 * g + w];
  uint4* cdst = reinterpret_cast<uint4*>(codes_base + row * (D / 2));
#pragma unroll
  for (int q = 0; q < D / 32; ++q) cdst[q] = make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
  if (TQ || D == 128)  // TQ4: the fp32 norm; FP4: D/32 scale bytes
    *reinterpret_cast<uint32_t*>(scales_base + row * 4) = static_cast<uint32_t>(scales);
  else if (D == 256)
    *reinterpret_cast<uint2*>(scales_base + row * 8) =
        make_uint2(static_cast<uint32_t>(scales), static_cast<uint32_t>(scales >> 32));
  else
    *reinterpret_cast<uint16_t*>(scales_base + row * 2) = static_cast<uint16_t>(scales);
}

// Quantiser stage of either format, then the store of the row.
template <int D, bool TQ>
__device__ __forceinline__ void quantize_store(float (&u)[D], const AppendParams& p, bool is_v, int64_t dst) {
  uint32_t codes[D / 8];
  uint64_t scales;
  if (TQ) {
    uint32_t norm_bits;
    quantize_tq_regs<D>(u, codes, norm_bits, p.tq_tpos);
    scales = norm_bits;
  } else {
    quantize_regs<D>(u, codes, scales, p.c);
  }
  if (is_v)
    store_row<D, false, TQ>(p.vc, p.vs, dst, codes, scales);
  else
    store_row<D, true, TQ>(p.kc, p.ks, dst, codes, scales);
}

template <int D, bool F32, bool TQ>
__global__ void __launch_bounds__(kAppendThreads)
    fp4_append_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                      const __grid_constant__ AppendParams p) {
  constexpr int ESZ = F32 ? 4 : 2;
  constexpr int ROWB = D * ESZ;          // bytes per input row
  constexpr int NBOX = ROWB / 128;       // 128-byte TMA boxes per row
  constexpr int BOXE = 128 / ESZ;        // elements per box row
  constexpr int TILEB = kRows * ROWB;    // one tensor, one stage
  constexpr int STAGEB = 2 * TILEB;      // K + V

  constexpr int NS = kAppendStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[NS];
  __shared__ int abort_flag;
  // The 128-byte swizzle pattern repeats every 1024 bytes: align the ring.
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int tid = threadIdx.x;
  const int64_t nrows = p.ntok * p.hkv;
  const int64_t ntiles = (nrows + kRows - 1) / kRows;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();

  auto issue = [&](int64_t tile, int stage) {
    uint8_t* st = smem + stage * STAGEB;
    mbar_arrive_expect_tx(&bars[stage], STAGEB);
    const int y = static_cast<int>(tile * kRows);
#pragma unroll
    for (int bx = 0; bx < NBOX; ++bx) {
      tma_load_2d(st + bx * kRows * 128, &mk, bx * BOXE, y, &bars[stage]);
      tma_load_2d(st + TILEB + bx * kRows * 128, &mv, bx * BOXE, y, &bars[stage]);
    }
  };

  const bool is_v = tid >= kRows;
  const int row = tid & (kRows - 1);
  int64_t tile = blockIdx.x;
  uint32_t it = 0;
  if (tid == 0)
    for (int s = 0; s < NS - 1; ++s)
      if (tile + static_cast<int64_t>(s) * gridDim.x < ntiles) issue(tile + static_cast<int64_t>(s) * gridDim.x, s);
  for (; tile < ntiles; tile += gridDim.x, ++it) {
    const int stage = it % NS;
    // the stage of the previous iteration is free again: it takes the tile NS - 1 ahead
    const int64_t ahead = tile + static_cast<int64_t>(NS - 1) * gridDim.x;
    if (tid == 0 && ahead < ntiles) issue(ahead, (it + NS - 1) % NS);
    const int64_t R = tile * kRows + row;
    // the row's token and its slot, read before the stage wait so that the
    // global load's latency passes during the wait and the rotation
    const int64_t t = R < nrows ? R / p.hkv : 0;
    const int64_t slot = R < nrows ? __ldg(p.slots + t) : -1;
    const bool ok = mbar_wait(&bars[stage], (it / NS) & 1, kWaitBudget);
    if (!ok) {
      record_error(p.status, kErrTimeout);
      abort_flag = 1;
    } else if (R < nrows) {
      const uint8_t* base = smem + stage * STAGEB + (is_v ? TILEB : 0) + row * 128;
      float u[D];
#pragma unroll
      for (int j = 0; j < ROWB / 16; ++j) {
        const int bx = j >> 3, cc = j & 7;
        const uint4 w = *reinterpret_cast<const uint4*>(base + bx * kRows * 128 + ((cc ^ (row & 7)) << 4));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        if (F32) {
#pragma unroll
          for (int k = 0; k < 4; ++k) u[4 * j + k] = __uint_as_float(ws[k] ^ p.sign.m[4 * j + k]);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            u[8 * j + 2 * k] = __uint_as_float((ws[k] << 16) ^ p.sign.m[8 * j + 2 * k]);
            u[8 * j + 2 * k + 1] = __uint_as_float((ws[k] & 0xFFFF0000u) ^ p.sign.m[8 * j + 2 * k + 1]);
          }
        }
      }
      rotate_regs<D>(u);
      const int h = static_cast<int>(R - t * p.hkv);
      if (slot >= p.num_slots) {
        record_error(p.status, kErrBounds);
      } else if (slot >= 0) {
        const int64_t page = slot >> p.ps_log2;
        const int64_t dst = ((page * p.hkv + h) << p.ps_log2) + (slot & ((1 << p.ps_log2) - 1));
        quantize_store<D, TQ>(u, p, is_v, dst);
      }
    }
    __syncthreads();
    if (abort_flag) {
      // Let copies that may still be in flight land before the block exits.
      if (tid == 0)
        for (int k = 0; k < NS; ++k)
          if (blockIdx.x + static_cast<int64_t>(it + k) * gridDim.x < ntiles)
            mbar_wait(&bars[(it + k) % NS], ((it + k) / NS) & 1, kWaitBudget);
      break;
    }
  }
}

// Small appends (a decode step's new tokens): one thread per K or V row read
// straight from global memory, no tensor maps -- the per-call host work of the
// tiled kernel would cost more than the copy.
template <int D, bool F32, bool TQ>
__global__ void __launch_bounds__(128) fp4_append_small_kernel(const void* k, const void* v,
                                                               const __grid_constant__ AppendParams p) {
  pdl_wait();
  const int64_t nrows = p.ntok * p.hkv;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= 2 * nrows) return;
  const bool is_v = gid >= nrows;
  const int64_t R = is_v ? gid - nrows : gid;
  float u[D];
  if (F32) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const float*>(is_v ? v : k) + R * D);
#pragma unroll
    for (int j = 0; j < D / 4; ++j) {
      const uint4 w = src[j];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) u[4 * j + e] = __uint_as_float(ws[e] ^ p.sign.m[4 * j + e]);
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(is_v ? v : k) + R * D);
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      const uint4 w = src[j];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        u[8 * j + 2 * e] = __uint_as_float((ws[e] << 16) ^ p.sign.m[8 * j + 2 * e]);
        u[8 * j + 2 * e + 1] = __uint_as_float((ws[e] & 0xFFFF0000u) ^ p.sign.m[8 * j + 2 * e + 1]);
      }
    }
  }
  rotate_regs<D>(u);
  const int64_t t = R / p.hkv;
  const int h = static_cast<int>(R - t * p.hkv);
  const int64_t slot = p.slots[t];
  if (slot >= p.num_slots) {
    record_error(p.status, kErrBounds);
  } else if (slot >= 0) {
    const int64_t page = slot >> p.ps_log2;
    const int64_t dst = ((page * p.hkv + h) << p.ps_log2) + (slot & ((1 << p.ps_log2) - 1));
    quantize_store<D, TQ>(u, p, is_v, dst);
  }
  pdl_trigger();
}

// D = 256 (FP4): one warp per row of K or V, since a 256-element row is too
// long for one thread's registers.  Lane l holds elements 8l .. 8l+7: the
// butterfly strides 1, 2, 4 run inside the lane, 8 .. 128 across lanes
// (partner l ^ (stride / 8)), each output with the same fp32 operations in the
// same ascending order as the one-thread rotation; a 32-channel group is 4
// lanes.  K rows keep the group-interleaved word order (word w of group g at
// word position 8 w + g).
template <bool F32>
__global__ void __launch_bounds__(128) fp4_append_wide_kernel(const void* k, const void* v,
                                                              const __grid_constant__ AppendParams p) {
  constexpr int D = 256;
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nrows = p.ntok * p.hkv;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (gw >= 2 * nrows) return;  // warp-uniform
  const bool is_v = gw >= nrows;
  const int64_t R = is_v ? gw - nrows : gw;
  const int64_t t = R / p.hkv;
  const int h = static_cast<int>(R - t * p.hkv);
  const int64_t slot = p.slots[t];
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (lane == 0) record_error(p.status, kErrBounds);
    return;
  }
  float u[8];
  if (F32) {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(is_v ? v : k) + R * D + 8 * lane);
    const float4 a = src[0], b = src[1];
    const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) u[e] = __uint_as_float(__float_as_uint(x[e]) ^ p.sign.m[8 * lane + e]);
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(is_v ? v : k) + R * D + 8 * lane);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      u[2 * e] = __uint_as_float((ws[e] << 16) ^ p.sign.m[8 * lane + 2 * e]);
      u[2 * e + 1] = __uint_as_float((ws[e] & 0xFFFF0000u) ^ p.sign.m[8 * lane + 2 * e + 1]);
    }
  }
#pragma unroll
  for (int hs = 1; hs < 8; hs <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & hs) == 0) {
        const float a = u[i], b = u[i + hs];
        u[i] = a + b;
        u[i + hs] = a - b;
      }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float o = __shfl_xor_sync(kFull, u[e], m);
      u[e] = upper ? (o - u[e]) : (u[e] + o);
    }
  }
  const float sc = inv_sqrt_d<D>();
#pragma unroll
  for (int e = 0; e < 8; ++e) u[e] *= sc;
  // group absmax over the group's 4 lanes, scale byte, codes
  float mx = max_abs_nan(u[0], u[1]);
#pragma unroll
  for (int e = 2; e < 8; ++e) mx = max_abs_nan(mx, u[e]);
  mx = max_abs_nan(mx, __shfl_xor_sync(kFull, mx, 1));
  mx = max_abs_nan(mx, __shfl_xor_sync(kFull, mx, 2));
  const uint32_t byte = scale_byte(fabsf(mx), p.c);
  const float inv = inv_scale(byte == 0xFFu ? 127u : byte);
#pragma unroll
  for (int e = 0; e < 8; ++e) u[e] *= inv;
  uint32_t word = cvt_e2m1x2(u[0], u[1]) | (cvt_e2m1x2(u[2], u[3]) << 8) | (cvt_e2m1x2(u[4], u[5]) << 16) |
                  (cvt_e2m1x2(u[6], u[7]) << 24);
  if (byte == 0xFFu) word = 0u;
  const int64_t page = slot >> p.ps_log2;
  const int64_t dst = ((page * p.hkv + h) << p.ps_log2) + (slot & ((1 << p.ps_log2) - 1));
  const int g = lane >> 2, w = lane & 3;
  uint32_t* crow = reinterpret_cast<uint32_t*>((is_v ? p.vc : p.kc) + dst * (D / 2));
  crow[is_v ? lane : (D / 32) * w + g] = word;
  if (w == 0) (is_v ? p.vs : p.ks)[dst * (D / 32) + g] = static_cast<uint8_t>(byte);
  pdl_trigger();
}

// ------------------------------------------------------------ FP8 / BF16
struct AnchorParams {
  const void* k;
  const void* v;
  const int64_t* slots;
  int64_t ntok;
  int hkv;
  int d;
  int ps_log2;
  int64_t num_slots;
  int fp8;  // 1: e4m3(x / scale), 0: bf16
  int in_fp32;
  float k_scale, v_scale;
  uint8_t* kc;
  uint8_t* vc;
  unsigned int* status;
};

// One thread per 8 consecutive elements of one row of K or V.
__global__ void __launch_bounds__(256) anchor_append_kernel(const __grid_constant__ AnchorParams p) {
  const int per_row = p.d / 8;
  const int64_t nrows = p.ntok * p.hkv;
  const int64_t total = 2 * nrows * per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int is_v = i >= nrows * per_row;
    const int64_t j = is_v ? i - nrows * per_row : i;
    const int64_t R = j / per_row;
    const int chunk = static_cast<int>(j - R * per_row);
    const int64_t t = R / p.hkv;
    const int h = static_cast<int>(R - t * p.hkv);
    const int64_t slot = p.slots[t];
    if (slot < 0) continue;
    if (slot >= p.num_slots) {
      record_error(p.status, kErrBounds);
      continue;
    }
    float x[8];
    const void* src = is_v ? p.v : p.k;
    if (p.in_fp32) {
      const float4* s4 = reinterpret_cast<const float4*>(static_cast<const float*>(src) + R * p.d + chunk * 8);
      const float4 a = s4[0], b = s4[1];
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
      const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + R * p.d + chunk * 8);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(ws[k] << 16);
        x[2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
      }
    }
    const int64_t page = slot >> p.ps_log2;
    const int64_t dst = ((page * p.hkv + h) << p.ps_log2) + (slot & ((1 << p.ps_log2) - 1));
    uint8_t* base = is_v ? p.vc : p.kc;
    if (p.fp8) {
      const float sc = is_v ? p.v_scale : p.k_scale;
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int k = 0; k < 4; k += 2) {
        lo |= cvt_e4m3x2(__fdiv_rn(x[k], sc), __fdiv_rn(x[k + 1], sc)) << (8 * k);
        hi |= cvt_e4m3x2(__fdiv_rn(x[4 + k], sc), __fdiv_rn(x[5 + k], sc)) << (8 * k);
      }
      *reinterpret_cast<uint2*>(base + dst * p.d + chunk * 8) = make_uint2(lo, hi);
    } else {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t*>(&b2);
      }
      *reinterpret_cast<uint4*>(base + (dst * p.d + chunk * 8) * 2) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// ------------------------------------------------------------ test kernels
template <int D>
__global__ void test_rotate_kernel(const float* x, int64_t n, float* y, const __grid_constant__ uqh::SignMasks sm) {
  const int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (r >= n) return;
  float u[D];
#pragma unroll
  for (int i = 0; i < D; ++i) u[i] = __uint_as_float(__float_as_uint(x[r * D + i]) ^ sm.m[i]);
  rotate_regs<D>(u);
#pragma unroll
  for (int i = 0; i < D; ++i) y[r * D + i] = u[i];
}

template <int D>
__global__ void test_quantize_kernel(const float* y, int64_t n, uint8_t* codes, uint8_t* scales) {
  const int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (r >= n) return;
  float u[D];
#pragma unroll
  for (int i = 0; i < D; ++i) u[i] = y[r * D + i];
  uint32_t c[D / 8];
  uint64_t s;
  quantize_regs<D>(u, c, s);
  store_row<D, false>(codes, scales, r, c, s);
}

// c calibration: the squared reconstruction error of the FP4 round trip of
// rotated rows, for each constant c of a list ([UQ-residency]: c* = argmin_c
// E[(z - c m q(z / (c m)))^2]; [UQ-review] §7.3: per-layer constants).  One
// thread per row: the row is rotated as in the append, then for each c every
// 32-channel group is coded with mode 0, the deployed rule (the append's scale
// byte, r = y * 2^-E and the hardware E2M1 conversion), or mode -1, a
// continuous scale s = c * m (r = fl32(y / s)); the error y - s * value is
// summed in fp64 and added to sse[c] once per warp.
struct CalibParams {
  const void* x;
  int64_t n;
  int in_fp32, n_c, mode;
  float c[64];
  double* sse;
  uqh::SignMasks sign;
};

template <int D>
__global__ void __launch_bounds__(128) calibrate_kernel(const __grid_constant__ CalibParams p) {
  const int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const bool live = r < p.n;
  float y[D];
#pragma unroll
  for (int i = 0; i < D; ++i) {
    uint32_t b = 0;
    if (live)
      b = p.in_fp32 ? __float_as_uint(static_cast<const float*>(p.x)[r * D + i])
                    : static_cast<uint32_t>(static_cast<const uint16_t*>(p.x)[r * D + i]) << 16;
    y[i] = __uint_as_float(b ^ p.sign.m[i]);
  }
  rotate_regs<D>(y);
  for (int ci = 0; ci < p.n_c; ++ci) {
    const float c = p.c[ci];
    double acc = 0.0;
#pragma unroll
    for (int g = 0; g < D / 32; ++g) {
      float mx = max_abs_nan(y[32 * g], y[32 * g + 1]);
#pragma unroll
      for (int i = 2; i < 32; ++i) mx = max_abs_nan(mx, y[32 * g + i]);
      const float m = fabsf(mx);
      if (m == 0.f) continue;
      uint32_t byte = 0;
      double s;
      float inv;
      if (p.mode == 0) {
        byte = scale_byte(m, c);
        s = ldexp(1.0, static_cast<int>(byte) - 127);
        inv = inv_scale(byte == 0xFFu ? 127u : byte);
      } else {
        s = static_cast<double>(c) * static_cast<double>(m);
        inv = 0.f;
      }
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        float e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float v = y[32 * g + 8 * w + k];
          e[k] = p.mode == 0 ? v * inv : static_cast<float>(static_cast<double>(v) / s);
        }
        const uint32_t word = cvt_e2m1x2(e[0], e[1]) | (cvt_e2m1x2(e[2], e[3]) << 8) |
                              (cvt_e2m1x2(e[4], e[5]) << 16) | (cvt_e2m1x2(e[6], e[7]) << 24);
        uint32_t h[4];
        e2m1x8_to_f16x2(word, h);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[k]));
          const double d0 = static_cast<double>(y[32 * g + 8 * w + 2 * k]) - static_cast<double>(f.x) * s;
          const double d1 = static_cast<double>(y[32 * g + 8 * w + 2 * k + 1]) - static_cast<double>(f.y) * s;
          acc += d0 * d0 + d1 * d1;
        }
      }
      if (byte == 0xFFu) acc = __longlong_as_double(0x7FF8000000000000ll);  // a non-finite group
    }
    if (!live) acc = 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(&p.sse[ci], acc);
  }
}

__global__ void test_cvt_e4m3_kernel(const float* x, int64_t n2, uint16_t* out) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i < n2) out[i] = static_cast<uint16_t>(cvt_e4m3x2(x[2 * i], x[2 * i + 1]));
}

// Stage hooks for R3 and R2 alone: the append's own conversion and scale-byte
// device functions applied to raw values.
__global__ void test_cvt_e2m1_kernel(const float* r, int64_t n2, uint8_t* out) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i < n2) {
    const uint32_t b = cvt_e2m1x2(r[2 * i], r[2 * i + 1]);
    out[2 * i] = static_cast<uint8_t>(b & 15u);
    out[2 * i + 1] = static_cast<uint8_t>(b >> 4);
  }
}

__global__ void test_scale_byte_kernel(const float* m, int64_t n, uint8_t* out) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i < n) out[i] = static_cast<uint8_t>(scale_byte(fabsf(m[i])));
}

// ------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Rows of `row_elems` elements, boxes of 128 bytes x kRows rows, 128-byte swizzle.
bool encode_rows(CUtensorMap* m, const void* base, int64_t rows, int row_elems, bool f32) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int esz = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_elems), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_elems) * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(kRows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool F32, bool TQ>
uq_status run_fp4_append(const CUtensorMap& mk, const CUtensorMap& mv, const AppendParams& p, int64_t nrows,
                         cudaStream_t s) {
  constexpr int STAGEB = 2 * kRows * D * (F32 ? 4 : 2);
  constexpr size_t smem = kAppendStages * STAGEB + 1024;
  auto kern = fp4_append_kernel<D, F32, TQ>;
  // The shared-memory attribute is per device and kernel: set once per device, with the
  // blocks per SM it allows (host threads may call concurrently).
  static std::mutex cfg_mu;
  static int cfg_per_sm[uqh::kMaxDevices];
  const uqh::DevInfo& di = uqh::dev_info();
  if (di.device < 0) return UQ_ERR_CUDA;
  int per_sm;
  {
    std::lock_guard<std::mutex> lk(cfg_mu);
    if (cfg_per_sm[di.device] == 0) {
      int n = 0;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kAppendThreads, smem) != cudaSuccess || n < 1)
        return UQ_ERR_CUDA;
      cfg_per_sm[di.device] = n;
    }
    per_sm = cfg_per_sm[di.device];
  }
  const int64_t ntiles = (nrows + kRows - 1) / kRows;
  const int64_t grid = std::min<int64_t>(ntiles, (int64_t)di.sms * per_sm);
  kern<<<(unsigned)grid, kAppendThreads, smem, s>>>(mk, mv, p);
  return uqh::cuda_status(cudaGetLastError());
}

}  // namespace

namespace uqh {

uq_status launch_append_fp4(const void* k, const void* v, bool in_fp32, int64_t ntok, const int64_t* slots,
                            const uq_cache& c, cudaStream_t s) {
  const int64_t nrows = ntok * c.num_kv_heads;
  if (nrows >= (int64_t(1) << 31) - kRows) return UQ_ERR_UNSUPPORTED;
  AppendParams p;
  p.slots = slots;
  p.ntok = ntok;
  p.hkv = c.num_kv_heads;
  p.ps_log2 = ilog2(c.page_size);
  p.num_slots = (int64_t)c.num_pages * c.page_size;
  p.kc = static_cast<uint8_t*>(c.k_codes);
  p.ks = static_cast<uint8_t*>(c.k_scales);
  p.vc = static_cast<uint8_t*>(c.v_codes);
  p.vs = static_cast<uint8_t*>(c.v_scales);
  p.status = status_word();
  make_sign_masks(c.rot_seed, c.head_dim, &p.sign);
  if (!p.status) return UQ_ERR_CUDA;
  const bool tq = c.dtype == UQ_TQ4;
  if (tq) {
    TqTables tt;
    const uq_status st = tq_tables(c.head_dim, &tt);
    if (st != UQ_OK) return st;
    for (int k = 0; k < 7; ++k) p.tq_tpos[k] = tt.tpos[k];
  } else {
    for (int k = 0; k < 7; ++k) p.tq_tpos[k] = 0.f;
  }
  p.c = fp4_c(c);
  if (c.head_dim == 256) {  // FP4 only: one warp per row, any size
    if (tq) return UQ_ERR_UNSUPPORTED;
    const unsigned grid = static_cast<unsigned>((2 * nrows + 3) / 4);
    return cuda_status(in_fp32 ? launch_pdl(fp4_append_wide_kernel<true>, grid, 128, 0, s, k, v, p)
                               : launch_pdl(fp4_append_wide_kernel<false>, grid, 128, 0, s, k, v, p));
  }
  // kernel instance by (head_dim, input type, format)
  const int which = (c.head_dim == 128 ? 4 : 0) + (in_fp32 ? 2 : 0) + (tq ? 1 : 0);
  if (nrows <= kSmallAppendRows) {
    const unsigned grid = static_cast<unsigned>((2 * nrows + 127) / 128);
    cudaError_t e;
    switch (which) {
      case 0: e = launch_pdl(fp4_append_small_kernel<64, false, false>, grid, 128, 0, s, k, v, p); break;
      case 1: e = launch_pdl(fp4_append_small_kernel<64, false, true>, grid, 128, 0, s, k, v, p); break;
      case 2: e = launch_pdl(fp4_append_small_kernel<64, true, false>, grid, 128, 0, s, k, v, p); break;
      case 3: e = launch_pdl(fp4_append_small_kernel<64, true, true>, grid, 128, 0, s, k, v, p); break;
      case 4: e = launch_pdl(fp4_append_small_kernel<128, false, false>, grid, 128, 0, s, k, v, p); break;
      case 5: e = launch_pdl(fp4_append_small_kernel<128, false, true>, grid, 128, 0, s, k, v, p); break;
      case 6: e = launch_pdl(fp4_append_small_kernel<128, true, false>, grid, 128, 0, s, k, v, p); break;
      default: e = launch_pdl(fp4_append_small_kernel<128, true, true>, grid, 128, 0, s, k, v, p); break;
    }
    return cuda_status(e);
  }
  CUtensorMap mk, mv;
  if (!encode_rows(&mk, k, nrows, c.head_dim, in_fp32) || !encode_rows(&mv, v, nrows, c.head_dim, in_fp32))
    return UQ_ERR_CUDA;
  switch (which) {
    case 0: return run_fp4_append<64, false, false>(mk, mv, p, nrows, s);
    case 1: return run_fp4_append<64, false, true>(mk, mv, p, nrows, s);
    case 2: return run_fp4_append<64, true, false>(mk, mv, p, nrows, s);
    case 3: return run_fp4_append<64, true, true>(mk, mv, p, nrows, s);
    case 4: return run_fp4_append<128, false, false>(mk, mv, p, nrows, s);
    case 5: return run_fp4_append<128, false, true>(mk, mv, p, nrows, s);
    case 6: return run_fp4_append<128, true, false>(mk, mv, p, nrows, s);
    default: return run_fp4_append<128, true, true>(mk, mv, p, nrows, s);
  }
}

uq_status launch_append_anchor(const void* k, const void* v, bool in_fp32, int64_t ntok, const int64_t* slots,
                               const uq_cache& c, cudaStream_t s) {
  AnchorParams p;
  p.k = k;
  p.v = v;
  p.slots = slots;
  p.ntok = ntok;
  p.hkv = c.num_kv_heads;
  p.d = c.head_dim;
  p.ps_log2 = ilog2(c.page_size);
  p.num_slots = (int64_t)c.num_pages * c.page_size;
  p.fp8 = c.dtype == UQ_FP8_E4M3;
  p.in_fp32 = in_fp32;
  p.k_scale = c.k_scale;
  p.v_scale = c.v_scale;
  p.kc = static_cast<uint8_t*>(c.k_codes);
  p.vc = static_cast<uint8_t*>(c.v_codes);
  p.status = status_word();
  if (!p.status) return UQ_ERR_CUDA;
  const int64_t work = 2 * ntok * c.num_kv_heads * (c.head_dim / 8);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, (int64_t)dev_info().sms * 8));
  anchor_append_kernel<<<(unsigned)grid, 256, 0, s>>>(p);
  return cuda_status(cudaGetLastError());
}

uq_status launch_test_rotate(const float* x, int64_t n, int d, uint64_t seed, float* y, cudaStream_t s) {
  SignMasks sm;
  make_sign_masks(seed, d, &sm);
  const unsigned grid = (unsigned)((n + 127) / 128);
  if (d == 256)
    test_rotate_kernel<256><<<grid, 128, 0, s>>>(x, n, y, sm);
  else if (d == 128)
    test_rotate_kernel<128><<<grid, 128, 0, s>>>(x, n, y, sm);
  else
    test_rotate_kernel<64><<<grid, 128, 0, s>>>(x, n, y, sm);
  return cuda_status(cudaGetLastError());
}

uq_status launch_test_quantize(const float* y, int64_t n, int d, uint8_t* codes, uint8_t* scales,
                               cudaStream_t s) {
  const unsigned grid = (unsigned)((n + 127) / 128);
  if (d == 256)
    test_quantize_kernel<256><<<grid, 128, 0, s>>>(y, n, codes, scales);
  else if (d == 128)
    test_quantize_kernel<128><<<grid, 128, 0, s>>>(y, n, codes, scales);
  else
    test_quantize_kernel<64><<<grid, 128, 0, s>>>(y, n, codes, scales);
  return cuda_status(cudaGetLastError());
}

uq_status launch_calibrate(const void* x, bool in_fp32, int64_t n, int d, uint64_t seed, const float* c_list,
                           int n_c, int mode, double* sse, cudaStream_t s) {
  CalibParams p;
  p.x = x;
  p.n = n;
  p.in_fp32 = in_fp32 ? 1 : 0;
  p.n_c = n_c;
  p.mode = mode;
  for (int i = 0; i < 64; ++i) p.c[i] = i < n_c ? c_list[i] : 0.f;
  p.sse = sse;
  make_sign_masks(seed, d, &p.sign);
  if (cudaMemsetAsync(sse, 0, sizeof(double) * n_c, s) != cudaSuccess) return UQ_ERR_CUDA;
  if (n == 0) return UQ_OK;
  const unsigned grid = static_cast<unsigned>((n + 127) / 128);
  if (d == 128)
    calibrate_kernel<128><<<grid, 128, 0, s>>>(p);
  else
    calibrate_kernel<64><<<grid, 128, 0, s>>>(p);
  return cuda_status(cudaGetLastError());
}

uq_status launch_test_cvt_e2m1(const float* r, int64_t n, uint8_t* out, cudaStream_t s) {
  const int64_t n2 = n / 2;
  test_cvt_e2m1_kernel<<<(unsigned)((n2 + 255) / 256), 256, 0, s>>>(r, n2, out);
  return cuda_status(cudaGetLastError());
}

uq_status launch_test_scale_byte(const float* m, int64_t n, uint8_t* out, cudaStream_t s) {
  test_scale_byte_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(m, n, out);
  return cuda_status(cudaGetLastError());
}

uq_status launch_test_cvt_e4m3(const float* x, int64_t n, uint8_t* out, cudaStream_t s) {
  const int64_t n2 = n / 2;
  test_cvt_e4m3_kernel<<<(unsigned)((n2 + 255) / 256), 256, 0, s>>>(x, n2, reinterpret_cast<uint16_t*>(out));
  return cuda_status(cudaGetLastError());
}

}  // namespace uqh
