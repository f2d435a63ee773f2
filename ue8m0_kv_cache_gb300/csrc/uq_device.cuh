// uq_device.cuh -- device building blocks shared by the append and decode
// kernels: packed-fp32 butterflies of the Walsh-Hadamard rotation, the UE8M0
// scale byte, FP4/FP8 conversions, and the mbarrier / bulk-copy (TMA) PTX.
//
// The rotation follows "UltraQuant: 4-bit KV Caching for Context-Heavy
// Agents" (review, manon006.tistory.com/395) §3.1: keys and values pass
// through a randomised Walsh-Hadamard transform before the 32-channel
// grouping.  Its fp32 arithmetic is fixed operation by operation so that the
// packed codes are reproducible bit for bit: signs applied first (exact),
// butterfly stages of stride 1, 2, 4, ... in that order, each output
// fl32(a+b) / fl32(a-b), then one multiply by fl32(1/sqrt(d)).  Packed
// add.f32x2 / sub.f32x2 perform the same IEEE round-to-nearest operations on
// two lanes at once, so they do not change any result.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace uqd {

constexpr unsigned kFull = 0xFFFFFFFFu;

// fl32(1/sqrt(d)) for the supported head dims.
template <int D>
__device__ __forceinline__ float inv_sqrt_d() {
  static_assert(D == 64 || D == 128 || D == 256, "head_dim");
  return D == 64 ? __uint_as_float(0x3E000000u) : D == 128 ? __uint_as_float(0x3DB504F3u) : __uint_as_float(0x3D800000u);
}

// (a, b) <- (a + b, a - b) on two lanes: (a0, b0) and (a1, b1).
__device__ __forceinline__ void bfly2(float& a0, float& a1, float& b0, float& b1) {
  asm("{\n\t.reg .b64 A, B, S, T;\n\t"
      "mov.b64 A, {%0, %1};\n\tmov.b64 B, {%2, %3};\n\t"
      "add.rn.f32x2 S, A, B;\n\tsub.rn.f32x2 T, A, B;\n\t"
      "mov.b64 {%0, %1}, S;\n\tmov.b64 {%2, %3}, T;\n\t}"
      : "+f"(a0), "+f"(a1), "+f"(b0), "+f"(b1));
}

// (a0, a1) += (b0, b1), round to nearest (one packed instruction).
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{\n\t.reg .b64 A, B;\n\tmov.b64 A, {%0, %1};\n\tmov.b64 B, {%2, %3};\n\t"
      "add.rn.f32x2 A, A, B;\n\tmov.b64 {%0, %1}, A;\n\t}"
      : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1));
}

// (a0, a1) = (b0, b1) * (s, s) + (a0, a1), round to nearest once.
__device__ __forceinline__ void fma2(float& a0, float& a1, float b0, float b1, float s) {
  asm("{\n\t.reg .b64 A, B, S;\n\tmov.b64 A, {%0, %1};\n\tmov.b64 B, {%2, %3};\n\t"
      "mov.b64 S, {%4, %4};\n\tfma.rn.f32x2 A, B, S, A;\n\tmov.b64 {%0, %1}, A;\n\t}"
      : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1), "f"(s));
}

// (a0, a1) * (s, s), round to nearest.
__device__ __forceinline__ void mul2(float& a0, float& a1, float s) {
  asm("{\n\t.reg .b64 A, S;\n\tmov.b64 A, {%0, %1};\n\tmov.b64 S, {%2, %2};\n\t"
      "mul.rn.f32x2 A, A, S;\n\tmov.b64 {%0, %1}, A;\n\t}"
      : "+f"(a0), "+f"(a1) : "f"(s));
}

// In-register Walsh-Hadamard butterflies over N consecutive elements, strides
// 1, 2, ..., N/2 in ascending order.  Stride 1 pairs two halves of one packed
// register and runs as scalar adds; every later stride runs packed.
template <int N>
__device__ __forceinline__ void fwht_regs(float (&u)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float a = u[i], b = u[i + 1];
    u[i] = a + b;
    u[i + 1] = a - b;
  }
#pragma unroll
  for (int h = 2; h < N; h <<= 1) {
#pragma unroll
    for (int i = 0; i < N; i += 2)
      if ((i & h) == 0) bfly2(u[i], u[i + 1], u[i + h], u[i + h + 1]);
  }
}

// Inverse rotation of one row spread over a warp, lane l holding elements
// l*EPL .. l*EPL+EPL-1 (EPL = D/32): o <- s .* fl32(FWHT_fp32(o) * fl32(1/sqrt D)),
// the transpose of the forward rotation (H is symmetric).  Butterfly strides
// ascend: those below EPL inside the lane, the rest across lanes by xor
// shuffles; the lower element of a pair becomes fl32(a+b), the upper fl32(a-b).
// sign_m[i] is the sign bit (0 or 0x80000000) of s_i.  Every lane must call it.
template <int D>
__device__ __forceinline__ void inverse_rotate_warp(float (&o)[D / 32], int lane, const uint32_t* sign_m) {
  constexpr int EPL = D / 32;
#pragma unroll
  for (int hs = 1; hs < EPL; hs <<= 1)
#pragma unroll
    for (int e = 0; e < EPL; ++e)
      if ((e & hs) == 0) {
        const float a = o[e], b = o[e + hs];
        o[e] = a + b;
        o[e + hs] = a - b;
      }
#pragma unroll
  for (int k = 1; k < 32; k <<= 1) {
    const bool upper = (lane & k) != 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float x = __shfl_xor_sync(kFull, o[e], k);
      o[e] = upper ? (x - o[e]) : (o[e] + x);
    }
  }
  const float sc = inv_sqrt_d<D>();
#pragma unroll
  for (int e = 0; e < EPL; ++e) o[e] = __uint_as_float(__float_as_uint(o[e] * sc) ^ sign_m[lane * EPL + e]);
}

// max(|a|, |b|) with NaN propagation (the sign of the result is meaningless;
// callers take fabsf at the end).
__device__ __forceinline__ float max_abs_nan(float a, float b) {
  float r;
  asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// UE8M0 byte of a group with absolute maximum m (m >= 0 or NaN):
// t = fl32(c * m), c = 0.156f unless a cache sets its own constant;
// E = integer nearest to log2(t); byte = clamp(E+127,
// 0, 254).  For a normal t = 2^(e-127) (1 + f/2^23), log2 t rounds up exactly
// when 1 + f/2^23 >= sqrt(2), i.e. f >= 0x3504F4 (sqrt(2) is irrational, so
// there are no ties).  A subnormal t = bits * 2^-149 rounds to 2^-126 (byte 1)
// when t >= 2^-126.5, i.e. bits >= 5931642; anything smaller clamps to 0.
// Non-finite m gives 0xFF.  (The 0.156 constant: [UQ-review] §3.3.)
constexpr float kFp4C = 0.156f;
__device__ __forceinline__ uint32_t scale_byte(float m, float c = kFp4C) {
  if (!(m <= 3.40282347e38f)) return 0xFFu;
  const float t = __fmul_rn(c, m);
  const uint32_t bits = __float_as_uint(t);
  if (bits >= 0x00800000u) {
    const uint32_t e = bits >> 23, f = bits & 0x7FFFFFu;
    const uint32_t b = e + (f >= 0x3504F4u ? 1u : 0u);
    return b > 254u ? 254u : b;
  }
  return bits >= 5931642u ? 1u : 0u;
}

// 2^-(byte-127) as fp32 (byte <= 254): exponent field 254 - byte, or the
// subnormal 2^-127 for byte 254.
__device__ __forceinline__ float inv_scale(uint32_t byte) {
  return byte <= 253u ? __uint_as_float((254u - byte) << 23) : __uint_as_float(0x00400000u);
}

// Two fp32 -> one byte of E2M1 codes, round to nearest even, saturating:
// low nibble = lo, high nibble = hi (the first source operand of the PTX
// conversion lands in the upper half).
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The four bytes of w, each a pair of E2M1 codes, to four f16x2 registers
// (hardware conversion; low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

// Two fp32 -> two E4M3 bytes (low byte = lo), round to nearest even, saturating.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 bytes (low byte -> low half) to f16x2; exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(r) : "r"(v));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t r;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(a));
  return r;
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B with a zero accumulator (the zero C operand needs no registers).
__device__ __forceinline__ void mma_f16_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One try_wait.  The suspend-time hint (in ns) lets the hardware park the
// thread until the phase completes (or the hint runs out) instead of having it
// spin on the barrier, which would take issue slots from the warps that work.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of the barrier for at most ~budget clock cycles.
// Returns false when the budget ran out (the caller records a timeout and
// winds down; nothing here can hang).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long budget) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > budget) return false;
  return true;
}

// 1-D bulk copy global -> shared (TMA engine), completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled tensor copy global -> shared (TMA), completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialisation attribute may start while the previous kernel in the
// stream is still running; it must wait for that kernel (and its memory) before
// touching global memory.  Without the attribute the wait returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream be scheduled (it still waits for this one to finish).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Record the first device-side error (1-based uq_status value) in the status word.
__device__ __forceinline__ void record_error(unsigned int* status, unsigned int code) {
  if (status) atomicCAS(status, 0u, code);
}

constexpr unsigned kErrTimeout = 6u;  // UQ_ERR_DEVICE_TIMEOUT
constexpr unsigned kErrBounds = 7u;   // UQ_ERR_DEVICE_BOUNDS
constexpr long long kWaitBudget = 4000000000ll;  // ~2 s at 2 GHz

// Cascade decode.  Group g holds the consecutive sequences cu[g] .. cu[g+1]-1,
// whose first prefix[g] keys are the same cache pages.  A group with at least
// min_rows query rows (sequences x query heads per kv head) has its first
// S_g = floor(min(prefix, cap) / 16) * 16 keys attended by the shared-prefix
// kernel, for all its sequences at once; the decode takes keys S_g .. L_b - 1
// of every sequence (from 16-token unit S_g / 16).  Other groups: S_g = 0.
__device__ __forceinline__ int casc_shared_keys(int nseq, int G, int prefix, int min_rows, int cap) {
  if (nseq <= 0 || prefix <= 0 || static_cast<long long>(nseq) * G < min_rows) return 0;
  return (prefix < cap ? prefix : cap) & ~15;
}

// The group g with cu[g] <= b < cu[g + 1], or -1 (cu non-decreasing over ng + 1 entries).
__device__ __forceinline__ int casc_group(const int32_t* cu, int ng, int b) {
  if (cu == nullptr || ng <= 0 || b < cu[0] || b >= cu[ng]) return -1;
  int lo = 0, hi = ng;  // cu[lo] <= b < cu[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= b) lo = mid; else hi = mid;
  }
  return b < cu[lo + 1] ? lo : -1;
}

}  // namespace uqd
