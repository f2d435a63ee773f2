// uq_decode.cu -- decode attention straight from the paged cache.
//
// The FP4 path follows "UltraQuant: 4-bit KV Caching for Context-Heavy
// Agents" (review, manon006.tistory.com/395): §3.2 the query is rotated into
// the key basis and rounded to FP8 E4M3, keys and values are consumed as
// E2M1 codes with UE8M0 group scales (value = code * 2^(byte-127)) and are
// never materialised as BF16 in memory; §4.2 the query is rounded once,
// outside the key-tile loop.  The output is rotated back (the rotation is
// orthogonal, "TurboQuant 완전 정리", inner-product preservation).
//
// GB300 design
//   * Work unit = 16 tokens of one (sequence, kv head, block of <= 8 query
//     heads).  All units of the batch are laid end to end and cut into equal
//     contiguous ranges, one per block of a persistent grid sized to the SMs,
//     so mixed sequence lengths stay balanced.  Each block writes one partial
//     (running max, sum, unnormalised output) per (sequence, kv head) range it
//     touches; a small merge kernel combines them by log-sum-exp and applies
//     the inverse rotation.
//   * Each of the 4 warps of a block streams its own units through a ring of
//     shared-memory stages on mbarriers: one unit = 16 rows of K codes, V
//     codes and their scale bytes (2176 bytes for head_dim 128), 136 bytes per
//     token-head.  FP4 and TQ4 stages are filled by per-lane 16-byte (codes)
//     and 4-byte (scales) cp.async copies; the FP8 and BF16 anchors' larger
//     rows by two 1-D bulk copies (TMA engine) per unit.
//   * QK^T and P.V run on the tensor cores as warp-level m16n8k16 f16 MMAs on
//     operands built in registers by the hardware e2m1x2 -> f16x2 conversion.
//     Keeping operands in registers avoids a second pass through shared
//     memory, which at n = 8 query heads would cap the kernel below HBM speed.
//   * QK^T runs one 32-channel group at a time into a fresh accumulator; the
//     group's UE8M0 scale is then applied to the fp32 partial logit, so K
//     values need no per-element scaling.  The cache stores K rows with the
//     groups interleaved by 4-byte words, so one 16-byte load gives each
//     thread one word of every group.
//   * P.V: V values of a thread all belong to one group, so its scale is one
//     packed half multiply; P is carried as hi + lo f16 parts (~22 bits) and
//     each 16-token unit is summed in a fresh accumulator before an IEEE fp32
//     add, so long contexts do not compound the accumulator's rounding.
//   * Sums over the head dimension do not depend on the order of channels,
//     so channels are assigned to fragment slots wherever the loads are
//     contiguous; the query and the output use the same assignment.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <cmath>

#include "uq_decode_common.cuh"
#include "uq_device.cuh"
#include "uq_internal.h"

namespace {

using namespace uqd;
using namespace uqdec;

// Softmax update for one unit: t[] are the log2-domain logits of tokens
// (r, r+8) x heads (2c, 2c+1).  Updates the running max / sum, rescales O when
// the max grows, and returns the P^T B fragments as hi/lo f16 parts of
// p * 2^15.
template <int NMMA>
__device__ __forceinline__ void softmax_unit(const float (&t)[4], float& M0, float& M1, float& L0, float& L1,
                                             float (&O)[NMMA][4], uint32_t (&bp)[4]) {
  // M does not have to be the exact max: p = 2^(t - M) stays exact for any M,
  // and the same M scales O and L.  It is raised (with a reduction of the
  // unit max across the 8 token rows and a rescale of O) only when some logit
  // exceeds it by more than kSlack, which after the first units is rare.
  float mc0 = fmaxf(t[0], t[2]), mc1 = fmaxf(t[1], t[3]);
  if (__any_sync(kFull, mc0 > M0 + kSlack || mc1 > M1 + kSlack)) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mc0 = fmaxf(mc0, __shfl_xor_sync(kFull, mc0, o));
      mc1 = fmaxf(mc1, __shfl_xor_sync(kFull, mc1, o));
    }
    const float n0 = fmaxf(M0, mc0), n1 = fmaxf(M1, mc1);
    const float a0 = ex2(M0 - n0), a1 = ex2(M1 - n1);
    M0 = n0;
    M1 = n1;
    L0 *= a0;
    L1 *= a1;
#pragma unroll
    for (int m = 0; m < NMMA; ++m) {
      O[m][0] *= a0; O[m][1] *= a1; O[m][2] *= a0; O[m][3] *= a1;
    }
  }
  const float s0 = kPShift - M0, s1 = kPShift - M1;
  const float p0 = ex2(t[0] + s0), p1 = ex2(t[1] + s1), p2 = ex2(t[2] + s0), p3 = ex2(t[3] + s1);
  L0 += p0 + p2;
  L1 += p1 + p3;
  // hi = p with the low 13 mantissa bits cleared (exact in f16), lo = the rest.
  const float h0 = __uint_as_float(__float_as_uint(p0) & 0xFFFFE000u);
  const float h1 = __uint_as_float(__float_as_uint(p1) & 0xFFFFE000u);
  const float h2 = __uint_as_float(__float_as_uint(p2) & 0xFFFFE000u);
  const float h3 = __uint_as_float(__float_as_uint(p3) & 0xFFFFE000u);
  // rows = tokens, cols = heads; transposed so that k = tokens.
  bp[0] = movmatrix_trans(pack_f16x2(h0, h1));
  bp[1] = movmatrix_trans(pack_f16x2(h2, h3));
  bp[2] = movmatrix_trans(pack_f16x2(p0 - h0, p1 - h1));
  bp[3] = movmatrix_trans(pack_f16x2(p2 - h2, p3 - h3));
}

// P.V of one 16-token unit for one 16-channel block into a fresh
// accumulator, then an IEEE fp32 add into the running output.
__device__ __forceinline__ void pv_unit(float (&o)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        const uint32_t (&bp)[4]) {
  float t[4];
  mma_f16_zc(t, a0, a1, a2, a3, bp[0], bp[1]);
  mma_f16(t, a0, a1, a2, a3, bp[2], bp[3]);
  add2(o[0], o[1], t[0], t[1]);
  add2(o[2], o[3], t[2], t[3]);
}

// Per-warp running state of one segment.
template <int NMMA>
struct WarpState {
  float M0, M1, L0, L1;
  float O[NMMA][4];
  uint32_t RV;   // FP4: reference exponent byte of O
  float rref;    // FP4: 2^(127 - RV)
  uint32_t bad;  // FP4: a non-finite group was seen
};

// NU consecutive units of this warp, FP4 cache, processed together: their
// QK^T chains are independent, the softmax bookkeeping (vote, rare reduction)
// is shared, and P.V accumulates all of them into one fresh accumulator per
// 16-channel block before the fp32 add.  TAIL: the last of the NU units may
// hold fewer than 16 valid tokens (a sequence's last unit); its masked tokens
// get logit -inf and value multiplier 0, whatever bytes their slots hold.
template <int D, int NU, bool TAIL>
__device__ __forceinline__ void units_fp4(const uint8_t* const (&st)[NU], int nvalid_last, int r, int c,
                                          const uint32_t (&qb)[D / 16][2], float sl2e, WarpState<D / 16>& S) {
  using C = DC<kFP4, D>;
  constexpr int NG = C::NG;
  constexpr int VB = C::VPT / 2;  // V code bytes per thread and token
  const int t0 = 2 * c, t1 = t0 + 1, t8 = t0 + 8, t9 = t0 + 9;

  // ---- QK^T per group: thread (r, c) holds word c of every group of tokens r, r+8
  float t[NU][4];
  uint32_t kbad = 0;
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const uint8_t* skc = st[u];
    const uint8_t* sks = st[u] + 2 * C::KBYTES;
    uint32_t kw0[NG], kw1[NG], ksw0, ksw1, ksw0b = 0u, ksw1b = 0u;  // scale bytes of groups 0-3 (b: 4-7)
    if (NG == 8) {  // D = 256: word c of the 8 groups is 32 contiguous bytes
      const uint4 a0 = *reinterpret_cast<const uint4*>(skc + r * C::KROW + c * 32);
      const uint4 b0 = *reinterpret_cast<const uint4*>(skc + r * C::KROW + c * 32 + 16);
      const uint4 a1 = *reinterpret_cast<const uint4*>(skc + (r + 8) * C::KROW + c * 32);
      const uint4 b1 = *reinterpret_cast<const uint4*>(skc + (r + 8) * C::KROW + c * 32 + 16);
      kw0[0] = a0.x; kw0[1] = a0.y; kw0[2 % NG] = a0.z; kw0[3 % NG] = a0.w;
      kw0[4 % NG] = b0.x; kw0[5 % NG] = b0.y; kw0[6 % NG] = b0.z; kw0[7 % NG] = b0.w;
      kw1[0] = a1.x; kw1[1] = a1.y; kw1[2 % NG] = a1.z; kw1[3 % NG] = a1.w;
      kw1[4 % NG] = b1.x; kw1[5 % NG] = b1.y; kw1[6 % NG] = b1.z; kw1[7 % NG] = b1.w;
      const uint2 s0 = *reinterpret_cast<const uint2*>(sks + r * 8);
      const uint2 s1 = *reinterpret_cast<const uint2*>(sks + (r + 8) * 8);
      ksw0 = s0.x; ksw0b = s0.y;
      ksw1 = s1.x; ksw1b = s1.y;
    } else if (NG == 4) {
      const uint4 x0 = *reinterpret_cast<const uint4*>(skc + r * C::KROW + c * 16);
      const uint4 x1 = *reinterpret_cast<const uint4*>(skc + (r + 8) * C::KROW + c * 16);
      kw0[0] = x0.x; kw0[1] = x0.y; kw0[2 % NG] = x0.z; kw0[3 % NG] = x0.w;
      kw1[0] = x1.x; kw1[1] = x1.y; kw1[2 % NG] = x1.z; kw1[3 % NG] = x1.w;
      ksw0 = *reinterpret_cast<const uint32_t*>(sks + r * 4);
      ksw1 = *reinterpret_cast<const uint32_t*>(sks + (r + 8) * 4);
    } else {
      const uint2 x0 = *reinterpret_cast<const uint2*>(skc + r * C::KROW + c * 8);
      const uint2 x1 = *reinterpret_cast<const uint2*>(skc + (r + 8) * C::KROW + c * 8);
      kw0[0] = x0.x; kw0[1 % NG] = x0.y;
      kw1[0] = x1.x; kw1[1 % NG] = x1.y;
      ksw0 = *reinterpret_cast<const uint16_t*>(sks + r * 2);
      ksw1 = *reinterpret_cast<const uint16_t*>(sks + (r + 8) * 2);
    }
    float sa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      uint32_t h0[4], h1[4];
      e2m1x8_to_f16x2(kw0[g], h0);
      e2m1x8_to_f16x2(kw1[g], h1);
      float acc[4];
      mma_f16_zc(acc, h0[0], h1[0], h0[1], h1[1], qb[2 * g][0], qb[2 * g][1]);
      mma_f16(acc, h0[2], h1[2], h0[3], h1[3], qb[2 * g + 1][0], qb[2 * g + 1][1]);
      float f0, f1;
      const uint32_t sw0 = g < 4 ? ksw0 : ksw0b, sw1 = g < 4 ? ksw1 : ksw1b;
      if ((g & 3) == 0) { f0 = scale_of<0>(sw0); f1 = scale_of<0>(sw1); }
      else if ((g & 3) == 1) { f0 = scale_of<1>(sw0); f1 = scale_of<1>(sw1); }
      else if ((g & 3) == 2) { f0 = scale_of<2>(sw0); f1 = scale_of<2>(sw1); }
      else { f0 = scale_of<3>(sw0); f1 = scale_of<3>(sw1); }
      fma2(sa[0], sa[1], acc[0], acc[1], f0);
      fma2(sa[2], sa[3], acc[2], acc[3], f1);
    }
    t[u][0] = sa[0] * sl2e; t[u][1] = sa[1] * sl2e; t[u][2] = sa[2] * sl2e; t[u][3] = sa[3] * sl2e;
    if (TAIL && u == NU - 1) {
      const bool v0 = r < nvalid_last, v1 = r + 8 < nvalid_last;
      if (!v0) { t[u][0] = -INFINITY; t[u][1] = -INFINITY; }
      if (!v1) { t[u][2] = -INFINITY; t[u][3] = -INFINITY; }
      kbad |= (v0 ? has_ff(ksw0) | has_ff(ksw0b) : 0u) | (v1 ? has_ff(ksw1) | has_ff(ksw1b) : 0u);
    } else {
      kbad |= has_ff(ksw0) | has_ff(ksw1) | has_ff(ksw0b) | has_ff(ksw1b);
    }
  }

  // ---- V scale bytes of the NU units (independent of QK^T; read before the
  // shared rare branch so that the branch splits the body only once)
  const int gv = (r * C::VPT) >> 5;
  uint32_t vb[NU][4];
  uint32_t bmax = 0;
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const uint8_t* svs = st[u] + 2 * C::KBYTES + C::SBYTES;
    vb[u][0] = svs[t0 * C::SROW + gv];
    vb[u][1] = svs[t1 * C::SROW + gv];
    vb[u][2] = svs[t8 * C::SROW + gv];
    vb[u][3] = svs[t9 * C::SROW + gv];
    if (TAIL && u == NU - 1) {
      if (t0 >= nvalid_last) vb[u][0] = 0;
      if (t1 >= nvalid_last) vb[u][1] = 0;
      if (t8 >= nvalid_last) vb[u][2] = 0;
      if (t9 >= nvalid_last) vb[u][3] = 0;
    }
    bmax = max(bmax, max(max(vb[u][0], vb[u][1]), max(vb[u][2], vb[u][3])));
  }
  S.bad |= kbad | (bmax == 0xFFu ? 1u : 0u);
  // Reference exponent RV = running max of the V scale bytes, so that every
  // multiplier 2^(byte - RV) is <= 1 and fits f16 together with the codes.
  const uint32_t RVc = __reduce_max_sync(kFull, bmax);

  // ---- softmax over the NU units
  float mc0 = -INFINITY, mc1 = -INFINITY;
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    mc0 = fmaxf(mc0, fmaxf(t[u][0], t[u][2]));
    mc1 = fmaxf(mc1, fmaxf(t[u][1], t[u][3]));
  }
  // One rare branch for both rescales of O: the running max M grew by more
  // than kSlack (after the first units, rare), or the V reference exponent
  // grew (rarer).  RVc and S.RV are warp-uniform.
  const bool grow_m = __any_sync(kFull, mc0 > S.M0 + kSlack || mc1 > S.M1 + kSlack);
  if (grow_m || RVc > S.RV) {
    float a0 = 1.f, a1 = 1.f, f = 1.f;
    if (grow_m) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mc0 = fmaxf(mc0, __shfl_xor_sync(kFull, mc0, o));
        mc1 = fmaxf(mc1, __shfl_xor_sync(kFull, mc1, o));
      }
      const float n0 = fmaxf(S.M0, mc0), n1 = fmaxf(S.M1, mc1);
      a0 = ex2(S.M0 - n0);
      a1 = ex2(S.M1 - n1);
      S.M0 = n0;
      S.M1 = n1;
      S.L0 *= a0;
      S.L1 *= a1;
    }
    if (RVc > S.RV) {
      f = pow2i(static_cast<int>(S.RV) - static_cast<int>(RVc));
      S.RV = RVc;
      S.rref = pow2i(127 - static_cast<int>(RVc));
    }
    a0 *= f;  // exact: f is a power of two
    a1 *= f;
#pragma unroll
    for (int m = 0; m < C::NMMA; ++m) {
      S.O[m][0] *= a0; S.O[m][1] *= a1; S.O[m][2] *= a0; S.O[m][3] *= a1;
    }
  }
  uint32_t bp[NU][4];
  {
    const float s0 = kPShift - S.M0, s1 = kPShift - S.M1;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const float p0 = ex2(t[u][0] + s0), p1 = ex2(t[u][1] + s1), p2 = ex2(t[u][2] + s0), p3 = ex2(t[u][3] + s1);
      S.L0 += p0 + p2;
      S.L1 += p1 + p3;
      const float h0 = __uint_as_float(__float_as_uint(p0) & 0xFFFFE000u);
      const float h1 = __uint_as_float(__float_as_uint(p1) & 0xFFFFE000u);
      const float h2 = __uint_as_float(__float_as_uint(p2) & 0xFFFFE000u);
      const float h3 = __uint_as_float(__float_as_uint(p3) & 0xFFFFE000u);
      bp[u][0] = movmatrix_trans(pack_f16x2(h0, h1));
      bp[u][1] = movmatrix_trans(pack_f16x2(h2, h3));
      bp[u][2] = movmatrix_trans(pack_f16x2(p0 - h0, p1 - h1));
      bp[u][3] = movmatrix_trans(pack_f16x2(p2 - h2, p3 - h3));
    }
  }

  // ---- P.V: thread (r, c) takes channels r*VPT.. of tokens 2c, 2c+1, 2c+8, 2c+9
  uint32_t mv01[NU], mv89[NU];
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    // 2^(byte-127) * 2^(127-RV), both exact powers of two (byte 0 gives 0).
    float f0 = __uint_as_float(vb[u][0] << 23) * S.rref, f1 = __uint_as_float(vb[u][1] << 23) * S.rref;
    float f8 = __uint_as_float(vb[u][2] << 23) * S.rref, f9 = __uint_as_float(vb[u][3] << 23) * S.rref;
    if (TAIL && u == NU - 1) {
      if (t0 >= nvalid_last) f0 = 0.f;
      if (t1 >= nvalid_last) f1 = 0.f;
      if (t8 >= nvalid_last) f8 = 0.f;
      if (t9 >= nvalid_last) f9 = 0.f;
    }
    mv01[u] = pack_f16x2(f0, f1);
    mv89[u] = pack_f16x2(f8, f9);
  }
#pragma unroll
  for (int q4 = 0; q4 < VB / 4; ++q4) {
    uint32_t A[NU][4][4];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const uint8_t* svc = st[u] + C::KBYTES;
      const uint32_t w0 = reinterpret_cast<const uint32_t*>(svc + t0 * C::KROW + r * VB)[q4];
      const uint32_t w1 = reinterpret_cast<const uint32_t*>(svc + t1 * C::KROW + r * VB)[q4];
      const uint32_t w8 = reinterpret_cast<const uint32_t*>(svc + t8 * C::KROW + r * VB)[q4];
      const uint32_t w9 = reinterpret_cast<const uint32_t*>(svc + t9 * C::KROW + r * VB)[q4];
      // Pair the same channel of two tokens in one byte (low nibble = lower token).
      e2m1x8_to_f16x2((w0 & 0x0F0F0F0Fu) | ((w1 & 0x0F0F0F0Fu) << 4), A[u][0]);
      e2m1x8_to_f16x2(((w0 >> 4) & 0x0F0F0F0Fu) | (w1 & 0xF0F0F0F0u), A[u][1]);
      e2m1x8_to_f16x2((w8 & 0x0F0F0F0Fu) | ((w9 & 0x0F0F0F0Fu) << 4), A[u][2]);
      e2m1x8_to_f16x2(((w8 >> 4) & 0x0F0F0F0Fu) | (w9 & 0xF0F0F0F0u), A[u][3]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float acc[4];
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        const uint32_t a0 = hmul2(A[u][0][k], mv01[u]), a1 = hmul2(A[u][1][k], mv01[u]);
        const uint32_t a2 = hmul2(A[u][2][k], mv89[u]), a3 = hmul2(A[u][3][k], mv89[u]);
        if (u == 0) mma_f16_zc(acc, a0, a1, a2, a3, bp[u][0], bp[u][1]);
        else mma_f16(acc, a0, a1, a2, a3, bp[u][0], bp[u][1]);
        mma_f16(acc, a0, a1, a2, a3, bp[u][2], bp[u][3]);
      }
      add2(S.O[4 * q4 + k][0], S.O[4 * q4 + k][1], acc[0], acc[1]);
      add2(S.O[4 * q4 + k][2], S.O[4 * q4 + k][3], acc[2], acc[3]);
    }
  }
}

// Byte permute with the PTX default mode: a selector nibble with bit 3 set
// replicates the sign bit of the selected byte over the result byte.
__device__ __forceinline__ uint32_t prmt_sx(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// TQ4 codebook lookup: the 8 sign-magnitude nibbles of w to 4 f16x2 (nibbles
// 2k, 2k+1 in o[k], low half first), the layout e2m1x8_to_f16x2 gives for FP4.
// lut[0..1] hold the high bytes of the f16 magnitudes c_0..c_7, lut[2..3] the
// low bytes: two byte permutes look up 4 magnitudes, two more interleave high
// and low bytes into f16 pairs, and one sign-replicating permute per pair
// moves the two sign bits (bit 3 of each nibble) to bits 15 and 31.
__device__ __forceinline__ void tq_lut8_to_f16x2(uint32_t w, const uint32_t (&lut)[4], uint32_t (&o)[4]) {
  const uint32_t sel = w & 0x77777777u;
  const uint32_t hb = __byte_perm(lut[0], lut[1], sel), lb = __byte_perm(lut[2], lut[3], sel);
  const uint32_t hb2 = __byte_perm(lut[0], lut[1], sel >> 16), lb2 = __byte_perm(lut[2], lut[3], sel >> 16);
  o[0] = __byte_perm(lb, hb, 0x5140);
  o[1] = __byte_perm(lb, hb, 0x7362);
  o[2] = __byte_perm(lb2, hb2, 0x5140);
  o[3] = __byte_perm(lb2, hb2, 0x7362);
  const uint32_t w4 = w << 4;  // bit 3 of nibble 2k becomes the top bit of byte k
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    // result byte 1 <- sign of byte k of w4 (nibble 2k), byte 3 <- sign of byte k of w (nibble 2k+1)
    const uint32_t s = prmt_sx(w, w4, ((0x8u | k) << 12) | ((0x8u | (4 + k)) << 4));
    o[k] ^= s & 0x80008000u;
  }
}

// NU consecutive units of this warp, TQ4 cache: the FP4 loop with codebook
// lookups in place of the hardware E2M1 conversion.  QK^T accumulates all
// groups in one accumulator and applies the key norm once; the value norm of
// each token is folded into P (times 2^(126 - RV), RV the running maximum of
// the norms' exponent fields, so that P stays within f16) instead of into the
// values.
template <int D, int NU, bool TAIL>
__device__ __forceinline__ void units_tq(const uint8_t* const (&st)[NU], int nvalid_last, int r, int c,
                                         const uint32_t (&qb)[D / 16][2], float sl2e, const uint32_t (&lut)[4],
                                         WarpState<D / 16>& S) {
  using C = DC<kTQ4, D>;
  constexpr int NG = C::NG;
  constexpr int VB = C::VPT / 2;  // V code bytes per thread and token
  const int t0 = 2 * c, t1 = t0 + 1, t8 = t0 + 8, t9 = t0 + 9;

  // ---- QK^T: thread (r, c) holds word c of every 32-channel group of tokens r, r+8
  float t[NU][4];
  uint32_t kbad = 0;
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const uint8_t* skc = st[u];
    const uint8_t* skn = st[u] + 2 * C::KBYTES;
    uint32_t kw0[NG], kw1[NG];
    if (NG == 4) {
      const uint4 x0 = *reinterpret_cast<const uint4*>(skc + r * C::KROW + c * 16);
      const uint4 x1 = *reinterpret_cast<const uint4*>(skc + (r + 8) * C::KROW + c * 16);
      kw0[0] = x0.x; kw0[1] = x0.y; kw0[2 % NG] = x0.z; kw0[3 % NG] = x0.w;
      kw1[0] = x1.x; kw1[1] = x1.y; kw1[2 % NG] = x1.z; kw1[3 % NG] = x1.w;
    } else {
      const uint2 x0 = *reinterpret_cast<const uint2*>(skc + r * C::KROW + c * 8);
      const uint2 x1 = *reinterpret_cast<const uint2*>(skc + (r + 8) * C::KROW + c * 8);
      kw0[0] = x0.x; kw0[1 % NG] = x0.y;
      kw1[0] = x1.x; kw1[1 % NG] = x1.y;
    }
    const float n0 = *reinterpret_cast<const float*>(skn + r * 4);
    const float n1 = *reinterpret_cast<const float*>(skn + (r + 8) * 4);
    float acc[4];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      uint32_t h0[4], h1[4];
      tq_lut8_to_f16x2(kw0[g], lut, h0);
      tq_lut8_to_f16x2(kw1[g], lut, h1);
      if (g == 0) mma_f16_zc(acc, h0[0], h1[0], h0[1], h1[1], qb[0][0], qb[0][1]);
      else mma_f16(acc, h0[0], h1[0], h0[1], h1[1], qb[2 * g][0], qb[2 * g][1]);
      mma_f16(acc, h0[2], h1[2], h0[3], h1[3], qb[2 * g + 1][0], qb[2 * g + 1][1]);
    }
    const float f0 = n0 * sl2e, f1 = n1 * sl2e;
    t[u][0] = acc[0] * f0; t[u][1] = acc[1] * f0; t[u][2] = acc[2] * f1; t[u][3] = acc[3] * f1;
    if (TAIL && u == NU - 1) {
      const bool v0 = r < nvalid_last, v1 = r + 8 < nvalid_last;
      if (!v0) { t[u][0] = -INFINITY; t[u][1] = -INFINITY; }
      if (!v1) { t[u][2] = -INFINITY; t[u][3] = -INFINITY; }
      kbad |= ((v0 && !(n0 <= 3.402823466e38f)) || (v1 && !(n1 <= 3.402823466e38f))) ? 1u : 0u;
    } else {
      kbad |= (!(n0 <= 3.402823466e38f) || !(n1 <= 3.402823466e38f)) ? 1u : 0u;
    }
  }

  // ---- V norms of tokens r, r+8 (the rows of this thread's P values)
  float vn[NU][2];
  uint32_t bmax = 0;
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const uint8_t* svn = st[u] + 2 * C::KBYTES + C::SBYTES;
    vn[u][0] = *reinterpret_cast<const float*>(svn + r * 4);
    vn[u][1] = *reinterpret_cast<const float*>(svn + (r + 8) * 4);
    if (TAIL && u == NU - 1) {
      if (r >= nvalid_last) vn[u][0] = 0.f;
      if (r + 8 >= nvalid_last) vn[u][1] = 0.f;
    }
    const uint32_t e0 = (__float_as_uint(vn[u][0]) >> 23) & 0xFFu, e1 = (__float_as_uint(vn[u][1]) >> 23) & 0xFFu;
    bmax = max(bmax, max(e0, e1));
  }
  S.bad |= kbad | (bmax == 0xFFu ? 1u : 0u);
  const uint32_t RVc = __reduce_max_sync(kFull, bmax);

  // ---- softmax, with the same shared rare branch as the FP4 path
  float mc0 = -INFINITY, mc1 = -INFINITY;
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    mc0 = fmaxf(mc0, fmaxf(t[u][0], t[u][2]));
    mc1 = fmaxf(mc1, fmaxf(t[u][1], t[u][3]));
  }
  const bool grow_m = __any_sync(kFull, mc0 > S.M0 + kSlack || mc1 > S.M1 + kSlack);
  if (grow_m || RVc > S.RV) {
    float a0 = 1.f, a1 = 1.f, f = 1.f;
    if (grow_m) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mc0 = fmaxf(mc0, __shfl_xor_sync(kFull, mc0, o));
        mc1 = fmaxf(mc1, __shfl_xor_sync(kFull, mc1, o));
      }
      const float n0 = fmaxf(S.M0, mc0), n1 = fmaxf(S.M1, mc1);
      a0 = ex2(S.M0 - n0);
      a1 = ex2(S.M1 - n1);
      S.M0 = n0;
      S.M1 = n1;
      S.L0 *= a0;
      S.L1 *= a1;
    }
    if (RVc > S.RV) {
      f = pow2i(static_cast<int>(S.RV) - static_cast<int>(RVc));
      S.RV = RVc;
      S.rref = pow2i(126 - static_cast<int>(RVc));
    }
    a0 *= f;
    a1 *= f;
#pragma unroll
    for (int m = 0; m < C::NMMA; ++m) {
      S.O[m][0] *= a0; S.O[m][1] *= a1; S.O[m][2] *= a0; S.O[m][3] *= a1;
    }
  }
  uint32_t bp[NU][4];
  {
    const float s0 = kPShift - S.M0, s1 = kPShift - S.M1;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const float p0 = ex2(t[u][0] + s0), p1 = ex2(t[u][1] + s1), p2 = ex2(t[u][2] + s0), p3 = ex2(t[u][3] + s1);
      S.L0 += p0 + p2;
      S.L1 += p1 + p3;
      // n * 2^(126 - RV) < 1 (exact: a power-of-two factor), then p * that
      const float w0 = vn[u][0] * S.rref, w1 = vn[u][1] * S.rref;
      const float q0 = p0 * w0, q1 = p1 * w0, q2 = p2 * w1, q3 = p3 * w1;
      const float h0 = __uint_as_float(__float_as_uint(q0) & 0xFFFFE000u);
      const float h1 = __uint_as_float(__float_as_uint(q1) & 0xFFFFE000u);
      const float h2 = __uint_as_float(__float_as_uint(q2) & 0xFFFFE000u);
      const float h3 = __uint_as_float(__float_as_uint(q3) & 0xFFFFE000u);
      bp[u][0] = movmatrix_trans(pack_f16x2(h0, h1));
      bp[u][1] = movmatrix_trans(pack_f16x2(h2, h3));
      bp[u][2] = movmatrix_trans(pack_f16x2(q0 - h0, q1 - h1));
      bp[u][3] = movmatrix_trans(pack_f16x2(q2 - h2, q3 - h3));
    }
  }

  // ---- P.V: thread (r, c) takes channels r*VPT.. of tokens 2c, 2c+1, 2c+8, 2c+9
#pragma unroll
  for (int q4 = 0; q4 < VB / 4; ++q4) {
    uint32_t A[NU][4][4];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const uint8_t* svc = st[u] + C::KBYTES;
      const uint32_t w0 = reinterpret_cast<const uint32_t*>(svc + t0 * C::KROW + r * VB)[q4];
      const uint32_t w1 = reinterpret_cast<const uint32_t*>(svc + t1 * C::KROW + r * VB)[q4];
      const uint32_t w8 = reinterpret_cast<const uint32_t*>(svc + t8 * C::KROW + r * VB)[q4];
      const uint32_t w9 = reinterpret_cast<const uint32_t*>(svc + t9 * C::KROW + r * VB)[q4];
      // same channel of two tokens in one byte (low nibble = lower token), then the lookup
      tq_lut8_to_f16x2((w0 & 0x0F0F0F0Fu) | ((w1 & 0x0F0F0F0Fu) << 4), lut, A[u][0]);
      tq_lut8_to_f16x2(((w0 >> 4) & 0x0F0F0F0Fu) | (w1 & 0xF0F0F0F0u), lut, A[u][1]);
      tq_lut8_to_f16x2((w8 & 0x0F0F0F0Fu) | ((w9 & 0x0F0F0F0Fu) << 4), lut, A[u][2]);
      tq_lut8_to_f16x2(((w8 >> 4) & 0x0F0F0F0Fu) | (w9 & 0xF0F0F0F0u), lut, A[u][3]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float acc[4];
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        if (u == 0) mma_f16_zc(acc, A[u][0][k], A[u][1][k], A[u][2][k], A[u][3][k], bp[u][0], bp[u][1]);
        else mma_f16(acc, A[u][0][k], A[u][1][k], A[u][2][k], A[u][3][k], bp[u][0], bp[u][1]);
        mma_f16(acc, A[u][0][k], A[u][1][k], A[u][2][k], A[u][3][k], bp[u][2], bp[u][3]);
      }
      add2(S.O[4 * q4 + k][0], S.O[4 * q4 + k][1], acc[0], acc[1]);
      add2(S.O[4 * q4 + k][2], S.O[4 * q4 + k][3], acc[2], acc[3]);
    }
  }
}

// One 16-token unit, FP8 or BF16 cache (unrotated, per-tensor scales folded
// into the logit scale and the final output).
template <int KIND, int D, bool TAIL>
__device__ __forceinline__ void unit_anchor(const uint8_t* st, int nvalid, int r, int c,
                                            const uint32_t (&qb)[D / 16][2], float fac,
                                            WarpState<D / 16>& S) {
  using C = DC<KIND, D>;
  const uint8_t* skc = st;
  const uint8_t* svc = st + C::KBYTES;
  float sacc[4] = {0.f, 0.f, 0.f, 0.f};
  if (KIND == kFP8) {
    const uint4* a0 = reinterpret_cast<const uint4*>(skc + r * C::KROW + c * C::CPT);
    const uint4* a1 = reinterpret_cast<const uint4*>(skc + (r + 8) * C::KROW + c * C::CPT);
#pragma unroll
    for (int q4 = 0; q4 < C::CPT / 16; ++q4) {
      const uint4 x0 = a0[q4], x1 = a1[q4];
      const uint32_t u0[4] = {x0.x, x0.y, x0.z, x0.w}, u1[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int m = 4 * q4 + k;
        mma_f16(sacc, e4m3x2_to_f16x2(u0[k]), e4m3x2_to_f16x2(u1[k]), e4m3x2_to_f16x2(u0[k] >> 16),
                e4m3x2_to_f16x2(u1[k] >> 16), qb[m][0], qb[m][1]);
      }
    }
  } else {
    const uint4* a0 = reinterpret_cast<const uint4*>(skc + r * C::KROW + c * C::CPT * 2);
    const uint4* a1 = reinterpret_cast<const uint4*>(skc + (r + 8) * C::KROW + c * C::CPT * 2);
#pragma unroll
    for (int q4 = 0; q4 < C::CPT / 8; ++q4) {
      const uint4 x0 = a0[q4], x1 = a1[q4];
      mma_bf16(sacc, x0.x, x1.x, x0.y, x1.y, qb[2 * q4][0], qb[2 * q4][1]);
      mma_bf16(sacc, x0.z, x1.z, x0.w, x1.w, qb[2 * q4 + 1][0], qb[2 * q4 + 1][1]);
    }
  }
  float t[4] = {sacc[0] * fac, sacc[1] * fac, sacc[2] * fac, sacc[3] * fac};
  if (TAIL) {
    if (r >= nvalid) { t[0] = -INFINITY; t[1] = -INFINITY; }
    if (r + 8 >= nvalid) { t[2] = -INFINITY; t[3] = -INFINITY; }
  }
  uint32_t bp[4];
  softmax_unit<C::NMMA>(t, S.M0, S.M1, S.L0, S.L1, S.O, bp);

  const int t0 = 2 * c, t1 = t0 + 1, t8 = t0 + 8, t9 = t0 + 9;
  const bool vt0 = !TAIL || t0 < nvalid, vt1 = !TAIL || t1 < nvalid;
  const bool vt8 = !TAIL || t8 < nvalid, vt9 = !TAIL || t9 < nvalid;
  if (KIND == kFP8) {
    constexpr int VB = C::VPT;  // bytes per thread and token
    uint32_t w0[VB / 4], w1[VB / 4], w8[VB / 4], w9[VB / 4];
#pragma unroll
    for (int q4 = 0; q4 < VB / 4; ++q4) {
      w0[q4] = vt0 ? reinterpret_cast<const uint32_t*>(svc + t0 * C::KROW + r * VB)[q4] : 0u;
      w1[q4] = vt1 ? reinterpret_cast<const uint32_t*>(svc + t1 * C::KROW + r * VB)[q4] : 0u;
      w8[q4] = vt8 ? reinterpret_cast<const uint32_t*>(svc + t8 * C::KROW + r * VB)[q4] : 0u;
      w9[q4] = vt9 ? reinterpret_cast<const uint32_t*>(svc + t9 * C::KROW + r * VB)[q4] : 0u;
    }
#pragma unroll
    for (int q4 = 0; q4 < VB / 4; ++q4) {
      const uint32_t x01 = __byte_perm(w0[q4], w1[q4], 0x5140), y01 = __byte_perm(w0[q4], w1[q4], 0x7362);
      const uint32_t x89 = __byte_perm(w8[q4], w9[q4], 0x5140), y89 = __byte_perm(w8[q4], w9[q4], 0x7362);
      pv_unit(S.O[2 * q4], e4m3x2_to_f16x2(x01), e4m3x2_to_f16x2(x01 >> 16), e4m3x2_to_f16x2(x89),
              e4m3x2_to_f16x2(x89 >> 16), bp);
      pv_unit(S.O[2 * q4 + 1], e4m3x2_to_f16x2(y01), e4m3x2_to_f16x2(y01 >> 16), e4m3x2_to_f16x2(y89),
              e4m3x2_to_f16x2(y89 >> 16), bp);
    }
  } else {
    constexpr int VW = C::VPT / 2;  // bf16 pairs per thread and token
    uint32_t w0[VW], w1[VW], w8[VW], w9[VW];
#pragma unroll
    for (int q4 = 0; q4 < VW; ++q4) {
      w0[q4] = vt0 ? reinterpret_cast<const uint32_t*>(svc + t0 * C::KROW + r * C::VPT * 2)[q4] : 0u;
      w1[q4] = vt1 ? reinterpret_cast<const uint32_t*>(svc + t1 * C::KROW + r * C::VPT * 2)[q4] : 0u;
      w8[q4] = vt8 ? reinterpret_cast<const uint32_t*>(svc + t8 * C::KROW + r * C::VPT * 2)[q4] : 0u;
      w9[q4] = vt9 ? reinterpret_cast<const uint32_t*>(svc + t9 * C::KROW + r * C::VPT * 2)[q4] : 0u;
    }
    auto bf2h = [](uint32_t w) {  // bf16x2 -> f16x2
      return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    };
#pragma unroll
    for (int m = 0; m < VW; ++m)
      pv_unit(S.O[m], bf2h(__byte_perm(w0[m], w1[m], 0x5410)), bf2h(__byte_perm(w0[m], w1[m], 0x7632)),
              bf2h(__byte_perm(w8[m], w9[m], 0x5410)), bf2h(__byte_perm(w8[m], w9[m], 0x7632)), bp);
  }
}

// Fused append: the warp that will take a sequence's last unit quantises that
// sequence's new token (position L - 1, physical slot new_slots[b]) itself --
// lanes 0-3 the K row, lanes 4-7 the V row of this kv head, with the append
// path's arithmetic -- and writes both rows to the cache and, in the stage's
// own layout, to a scratch row in shared memory.  It runs at the start of the
// segment, while the first copies are in flight; when the last unit's stage
// lands (its copy of that slot may predate the write), patch_stage puts the
// scratch row over the token's row.  So no separate append launch precedes
// the decode.  A slot that disagrees with the block table's position for the
// token is an error (recorded; nothing written, returns false).
template <int D>
__device__ __noinline__ bool fused_append(const DecParams& p, uint8_t* scratch, int b, int kvh, int L,
                                          const int32_t* bt_row, int lane) {
  using C = DC<kFP4, D>;
  constexpr int CPT = D / 4, NG = D / 32, NW = CPT / 8;  // channels, groups, code words per thread
  const int64_t slot = p.new_slots[b];
  if (slot < 0) return false;
  const int tok = L - 1;
  const int ps_mask = (1 << p.ps_log2) - 1;
  const int64_t bslot = tok < 0 ? -1 : (static_cast<int64_t>(bt_row[tok >> p.ps_log2]) << p.ps_log2) + (tok & ps_mask);
  if (slot != bslot || slot >= p.num_slots) {
    if (lane == 0) record_error(p.status, kErrBounds);
    return false;
  }
  const int quad = lane >> 2, c = lane & 3;
  const bool is_v = quad == 1, active = quad < 2;
  const size_t esz = p.new_f32 ? 4 : 2;
  const uint8_t* src = static_cast<const uint8_t*>(is_v ? p.v_new : p.k_new) +
                       (static_cast<int64_t>(b) * p.Hkv + kvh) * D * esz;
  float x[CPT];
  if (p.new_f32) rotate_quad<D, true>(src, active, c, p.sign, x);
  else rotate_quad<D, false>(src, active, c, p.sign, x);
  uint32_t codes[NW], byte;
  quantize_quad<D>(x, codes, byte, p.fp4_c);
  if (active) {
    const int64_t dst = (((slot >> p.ps_log2) * p.Hkv + kvh) << p.ps_log2) + (slot & ps_mask);
    uint8_t* gcodes = (is_v ? p.wvc : p.wkc) + dst * C::KROW;
    uint8_t* scodes = scratch + (is_v ? C::KROW : 0);
#pragma unroll
    for (int k = 0; k < NW; ++k) {
      const int nw = c * NW + k;                           // natural word index in the row
      const int pos = is_v ? nw : NG * (nw & 3) + (nw >> 2);  // K rows: group-interleaved words
      *reinterpret_cast<uint32_t*>(gcodes + 4 * pos) = codes[k];
      *reinterpret_cast<uint32_t*>(scodes + 4 * pos) = codes[k];
    }
    if (CPT == 32 || (c & 1) == 0) {
      const int g = c * CPT / 32;
      (is_v ? p.wvs : p.wks)[dst * NG + g] = static_cast<uint8_t>(byte);
      scratch[2 * C::KROW + (is_v ? C::SROW : 0) + g] = static_cast<uint8_t>(byte);
    }
  }
  __syncwarp();
  return true;
}

// Copies the scratch row written by fused_append over row r of a landed stage.
template <int D>
__device__ __forceinline__ void patch_stage(const uint8_t* scratch, uint8_t* st, int r, int lane) {
  using C = DC<kFP4, D>;
  constexpr int KW = C::KROW / 4;  // code words per row
  if (lane < 2 * KW) {
    const int v = lane >= KW, wd = lane - (v ? KW : 0);
    *reinterpret_cast<uint32_t*>(st + (v ? C::KBYTES : 0) + r * C::KROW + 4 * wd) =
        *reinterpret_cast<const uint32_t*>(scratch + (v ? C::KROW : 0) + 4 * wd);
  }
  if (lane < 2 * C::SROW) {
    const int v = lane >= C::SROW, g = lane - (v ? C::SROW : 0);
    st[2 * C::KBYTES + (v ? C::SBYTES : 0) + r * C::SROW + g] = scratch[2 * C::KROW + (v ? C::SROW : 0) + g];
  }
}

// The fused append on its own (one warp per (sequence, kv head)), run before
// the tensor-memory decode, which reads the new token from the cache.
template <int D>
__global__ void __launch_bounds__(32) append_step_kernel(const __grid_constant__ DecParams p) {
  __shared__ __align__(16) uint8_t scratch[2 * DC<kFP4, D>::KROW + 2 * DC<kFP4, D>::SROW];
  pdl_wait();
  const int b = blockIdx.x / p.Hkv, kvh = blockIdx.x - b * p.Hkv;
  const int L = clamp_len(p, b);
  fused_append<D>(p, scratch, b, kvh, L, p.block_table + static_cast<int64_t>(b) * p.max_pages, threadIdx.x);
  pdl_trigger();
}

template <int KIND, int D>
__global__ void __launch_bounds__(kThreads, D == 256 ? (packed4(KIND) ? 2 : 1) : (packed4(KIND) ? UQ_FP4_MINB : 4))
    decode_kernel(const __grid_constant__ DecParams p) {
  using C = DC<KIND, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * C::NST * C::STAGE);
  float* comb_ml = reinterpret_cast<float*>(bars + kWarps * C::NST);
  float* comb_o = comb_ml + kWarps * kHB * 2;
  int* pre = reinterpret_cast<int*>(comb_o + kWarps * kHB * D);
  __shared__ int abort_flag;
  __shared__ uint64_t stall_bar;  // injected timeout: nothing ever arrives at it

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane >> 2, c = lane & 3;
  const int ps_mask = (1 << p.ps_log2) - 1;
  uint32_t lut[4];  // TQ4 codebook byte tables
#pragma unroll
  for (int i = 0; i < 4; ++i) lut[i] = p.tq_lut[i];
  pdl_wait();  // the cache, query and block table are written by earlier kernels

  // Prefix sums of 16-token units per sequence.
  if (warp == 0) {
    int run = 0;
    if (lane == 0) pre[0] = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      int x = 0;
      if (b < p.B) {
        const int L = clamp_len(p, b), skip = casc_skip(p, b);
        if (skip > L) record_error(p.status, kErrBounds);  // a shared prefix longer than the sequence
        x = max(0, (L + kChunk - 1) / kChunk - skip / kChunk);
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      if (b < p.B) pre[b + 1] = run + x;
      run += __shfl_sync(kFull, x, 31);
    }
  }
  uint64_t* mybars = bars + warp * C::NST;
  uint8_t* myring = ring + warp * C::NST * C::STAGE;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < C::NST; ++s) mbar_init(&mybars[s], packed4(KIND) ? 32 : 1);  // see the copy issue
    fence_mbar_init();
  }
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&stall_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  bool stall = p.stall_cta == static_cast<int>(blockIdx.x) && warp == 0;  // warp-uniform

  const int pps = p.Hkv * p.nhb;  // (kv head, head block) pairs per sequence
  const int64_t U = static_cast<int64_t>(pre[p.B]) * pps;
  int64_t lo, hi;
  block_range(blockIdx.x, U, gridDim.x, lo, hi);
  if (blockIdx.x == 0 && tid == 0) *p.ws_units = U;
  uint32_t it = 0;  // position in this warp's ring, carried across segments

  for (int64_t u = lo; u < hi;) {
    // Segment: the units of one (sequence, kv head, head block) inside [u, hi).
    int lb = 1, hb_ = p.B;  // first index with pre[idx] * pps > u, in [1, B]
    while (lb < hb_) {
      const int mid = (lb + hb_) >> 1;
      if (static_cast<int64_t>(pre[mid]) * pps > u) hb_ = mid; else lb = mid + 1;
    }
    const int b = lb - 1;
    const int nb = pre[b + 1] - pre[b];
    const int64_t off = u - static_cast<int64_t>(pre[b]) * pps;
    const int pl = static_cast<int>(off / nb);
    const int j0 = static_cast<int>(off - static_cast<int64_t>(pl) * nb);
    const int seg = static_cast<int>((nb - j0) < (hi - u) ? (nb - j0) : (hi - u));
    const int kvh = pl / p.nhb, hblk = pl - kvh * p.nhb;
    const int pair = b * pps + pl;
    const int L = clamp_len(p, b);
    const int ub = casc_skip(p, b) / kChunk;  // first unit of the sequence that this decode takes

    // Query fragments (once per segment, outside the unit loop).
    uint32_t qb[C::NMMA][2];
    {
      const int hloc = hblk * kHB + r;
      const bool hv = hloc < p.G;
      const uint16_t* qrow = p.q + (static_cast<int64_t>(b) * p.Hq + kvh * p.G + (hv ? hloc : 0)) * D;
      if constexpr (KIND == kFP4) {
        // Rotate and round on the quad, then regroup through this warp's slice
        // of the combine buffer: thread c needs bytes 32g + 8c .. +7 of its
        // head for every group g (the fragment order of the QK^T loop).
        uint32_t qbytes[D / 16];
        rotated_query_bytes<D>(qrow, hv, c, p.sign, qbytes);
        uint8_t* qs = reinterpret_cast<uint8_t*>(comb_o + warp * kHB * D);
#pragma unroll
        for (int e = 0; e < D / 16; ++e) *reinterpret_cast<uint32_t*>(qs + r * D + c * (D / 4) + 4 * e) = qbytes[e];
        __syncwarp();
#pragma unroll
        for (int g = 0; g < C::NG; ++g) {
          const uint2 w = *reinterpret_cast<const uint2*>(qs + r * D + 32 * g + 8 * c);
          qb[2 * g][0] = e4m3x2_to_f16x2(w.x);
          qb[2 * g][1] = e4m3x2_to_f16x2(w.x >> 16);
          qb[2 * g + 1][0] = e4m3x2_to_f16x2(w.y);
          qb[2 * g + 1][1] = e4m3x2_to_f16x2(w.y >> 16);
        }
        __syncwarp();
      } else if constexpr (KIND == kTQ4) {
        // Rotate on the quad, round to f16 (nearest even), regroup through
        // the warp's slice of the combine buffer: thread c needs channels
        // 32g + 8c .. +7 of its head for every group g.
        float x[D / 4];
        rotate_quad<D, false>(qrow, hv, c, p.sign, x);
        uint32_t* qs = reinterpret_cast<uint32_t*>(comb_o + warp * kHB * D);  // [8 heads][D] f16
#pragma unroll
        for (int e = 0; e < D / 4; e += 2) qs[(r * D + c * (D / 4) + e) / 2] = pack_f16x2(x[e], x[e + 1]);
        __syncwarp();
#pragma unroll
        for (int g = 0; g < C::NG; ++g) {
          const uint4 w = *reinterpret_cast<const uint4*>(qs + (r * D + 32 * g + 8 * c) / 2);
          qb[2 * g][0] = w.x;
          qb[2 * g][1] = w.y;
          qb[2 * g + 1][0] = w.z;
          qb[2 * g + 1][1] = w.w;
        }
        __syncwarp();
      } else {
#pragma unroll
        for (int m = 0; m < C::NMMA; ++m) {
          const uint32_t x0 = hv ? *reinterpret_cast<const uint32_t*>(qrow + c * C::CPT + 4 * m) : 0u;
          const uint32_t x1 = hv ? *reinterpret_cast<const uint32_t*>(qrow + c * C::CPT + 4 * m + 2) : 0u;
          if (KIND == kBF16) {
            qb[m][0] = x0;
            qb[m][1] = x1;
          } else {  // bf16 -> f16 (exact for |q| in the f16 normal range)
            qb[m][0] = pack_f16x2(__uint_as_float(x0 << 16), __uint_as_float(x0 & 0xFFFF0000u));
            qb[m][1] = pack_f16x2(__uint_as_float(x1 << 16), __uint_as_float(x1 & 0xFFFF0000u));
          }
        }
      }
    }

    const int nw = seg > warp ? (seg - warp + kWarps - 1) / kWarps : 0;
    const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.max_pages;
    // Lane l holds the page of this warp's unit (32*k + l) in pf and of unit
    // (32*(k+1) + l) in pf_next; pf_next is loaded 32 units before it is
    // needed, so the copy issue never waits on a dependent global load.
    auto page_of_lane = [&](int i) {
      int page = 0;
      if (i < nw) {
        page = bt_row[((ub + j0 + warp + i * kWarps) * kChunk) >> p.ps_log2];
        if (page < 0 || page >= p.num_pages) {
          record_error(p.status, kErrBounds);
          page = 0;
        }
      }
      return page;
    };
    int pf = page_of_lane(lane), pf_next = page_of_lane(32 + lane);
    // FP4 and TQ4: every lane copies 16-byte chunks of the unit's K and V code
    // rows and 4-byte words of its scale (or norm) rows with cp.async, and one
    // no-increment arrival per lane completes the stage barrier (32 arrivals):
    // per-lane copies go through the load/store path at its full rate, where
    // each bulk-copy request would cost the copy engine a fixed issue time.
    // The anchors' larger rows (FP8 2 KB, BF16 4 KB per array and unit) come
    // by two bulk copies, from lanes 0 and 1, on a barrier of one arrival.
    const uint8_t* cp_base = lane == 1 ? p.vc : p.kc;
    const uint32_t cp_off = lane == 1 ? C::KBYTES : 0;
    const uint32_t ring_u32 = smem_u32(myring), bars_u32 = smem_u32(mybars);
    // FP4 / TQ4 per-lane copy sources and destinations, fixed for the segment:
    // lane l copies 16-byte chunks l, l + 32, ... of the unit's K and V code
    // rows and 4-byte word l (< 2 SW) of its two side rows.  Per unit only the
    // row offset changes: one wide multiply-add per array.
    constexpr int CW = C::KBYTES / 16;  // 16-byte chunks per array and unit
    constexpr int SW = C::SBYTES / 4;   // side words per array and unit
    static_assert(CW % 32 == 0 && (2 * SW) % 32 == 0 || (2 * SW) < 32, "copy split over the lanes");
    const uint8_t* kc_l = p.kc + 16 * lane;
    const uint8_t* vc_l = p.vc + 16 * lane;
    const uint8_t* sd_l = lane < SW ? p.ks + 4 * lane : p.vs + 4 * (lane - SW);
    const uint32_t dc_l = ring_u32 + 16 * lane, ds_l = ring_u32 + 2 * C::KBYTES + 4 * lane;
    const uint32_t rowh = static_cast<uint32_t>(kvh) << p.ps_log2;  // (page * Hkv + kvh) * ps = page * Hkv * ps + rowh
    const uint32_t page_rows = static_cast<uint32_t>(p.Hkv) << p.ps_log2;
    auto issue = [&](int i, int slot, int page) {
      const int tok0 = (ub + j0 + warp + i * kWarps) * kChunk;
      const uint32_t bar = bars_u32 + 8u * slot;
      if (packed4(KIND)) {
        // physical row of the unit's first token; < num_pages * Hkv * ps, checked on the host to fit 32 bits
        const uint32_t row = static_cast<uint32_t>(page) * page_rows + rowh + (tok0 & ps_mask);
        const uint8_t* gk = kc_l + static_cast<uint64_t>(row) * C::KROW;
        const uint8_t* gv = vc_l + static_cast<uint64_t>(row) * C::KROW;
        const uint32_t dst = dc_l + slot * uint32_t(C::STAGE);
#pragma unroll
        for (int j = 0; j < CW / 32; ++j) {
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 512 * j), "l"(gk + 512 * j)
                       : "memory");
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + C::KBYTES + 512 * j),
                       "l"(gv + 512 * j) : "memory");
        }
        const uint8_t* gs = sd_l + static_cast<uint64_t>(row) * C::SROW;
        const uint32_t ds = ds_l + slot * uint32_t(C::STAGE);
#pragma unroll
        for (int j = 0; j < (2 * SW) / 32; ++j) {  // head_dim 256: words 32..63 are the V side row
          const uint8_t* g = j == 0 ? gs : p.vs + static_cast<uint64_t>(row) * C::SROW + 4 * lane;
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(ds + 128 * j), "l"(g) : "memory");
        }
        if ((2 * SW) % 32 != 0 && lane < (2 * SW) % 32)
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(ds), "l"(gs) : "memory");
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
      } else {
        const int64_t row0 = ((static_cast<int64_t>(page) * p.Hkv + kvh) << p.ps_log2) + (tok0 & ps_mask);
        const uint32_t sbase = ring_u32 + slot * uint32_t(C::STAGE);
        if (lane == 0)
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                       "r"(uint32_t(2 * C::KBYTES)) : "memory");
        if (lane < 2)
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                  sbase + cp_off),
              "l"(cp_base + row0 * C::KROW), "r"(uint32_t(C::KBYTES)), "r"(bar)
              : "memory");
      }
    };
    for (int i = 0; i < (nw < C::NST ? nw : C::NST); ++i) issue(i, (it + i) % C::NST, __shfl_sync(kFull, pf, i));
    // The new token (fused append) is quantised while those copies fly; its
    // scratch row sits in this warp's slice of the combine buffer, past the
    // query bytes, which is free until the combine.
    int fa_unit = -1;  // index of the unit whose stage takes the scratch row
    uint8_t* fa_scratch = reinterpret_cast<uint8_t*>(comb_o + warp * kHB * D) + kHB * D;
    if constexpr (KIND == kFP4 && D <= 128) {  // the fused append (FP4, head dims 64 and 128)
      if (p.new_slots != nullptr && nw > 0 && j0 + warp + (nw - 1) * kWarps == nb - 1)
        if (fused_append<D>(p, fa_scratch, b, kvh, L, bt_row, lane)) fa_unit = nw - 1;
    }

    WarpState<C::NMMA> S;
    S.M0 = S.M1 = -INFINITY;
    S.L0 = S.L1 = 0.f;
    S.RV = 0;
    S.rref = pow2i(KIND == kTQ4 ? 126 : 127);
    S.bad = 0;
#pragma unroll
    for (int m = 0; m < C::NMMA; ++m) S.O[m][0] = S.O[m][1] = S.O[m][2] = S.O[m][3] = 0.f;
    const float fac = KIND == kFP8 ? p.sl2e * p.k_scale : p.sl2e;

    for (int i = 0; i < nw;) {
      // FP4 takes two units per step (independent work for the scheduler);
      // the anchors, and an odd last unit, take one.
      const int nu = (packed4(KIND) && i + 1 < nw) ? 2 : 1;  // warp-uniform
      bool ok = mbar_wait(&mybars[it % C::NST], (it / C::NST) & 1, kWaitBudget);
      if (nu == 2) ok = ok && mbar_wait(&mybars[(it + 1) % C::NST], ((it + 1) / C::NST) & 1, kWaitBudget);
      if (stall) {  // injected timeout (test hook): a bounded wait that runs out
        ok = ok && mbar_wait(&stall_bar, 0, p.stall_budget);
        stall = false;
      }
      if (!__all_sync(kFull, ok)) {
        if (lane == 0) {
          record_error(p.status, kErrTimeout);
          for (int k = i; k < (nw < i + C::NST ? nw : i + C::NST); ++k)
            mbar_wait(&mybars[(it + k - i) % C::NST], ((it + k - i) / C::NST) & 1, kWaitBudget);
        }
        abort_flag = 1;
        it += nw - i;
        break;
      }
      if constexpr (KIND == kFP4 && D <= 128) {
        if (fa_unit >= 0 && fa_unit - i < nu) {
          patch_stage<D>(fa_scratch, myring + ((it + fa_unit - i) % C::NST) * C::STAGE, (L - 1) & (kChunk - 1),
                         lane);
          fa_unit = -1;
          __syncwarp();
        }
      }
      const uint8_t* st0 = myring + (it % C::NST) * C::STAGE;
      const int nvalid = L - (ub + j0 + warp + (i + nu - 1) * kWarps) * kChunk;  // of the last unit taken
      if constexpr (KIND == kFP4) {
        if (nu == 2) {
          const uint8_t* const sts[2] = {st0, myring + ((it + 1) % C::NST) * C::STAGE};
          if (nvalid >= kChunk) units_fp4<D, 2, false>(sts, kChunk, r, c, qb, fac, S);
          else units_fp4<D, 2, true>(sts, nvalid, r, c, qb, fac, S);
        } else {
          const uint8_t* const sts[1] = {st0};
          if (nvalid >= kChunk) units_fp4<D, 1, false>(sts, kChunk, r, c, qb, fac, S);
          else units_fp4<D, 1, true>(sts, nvalid, r, c, qb, fac, S);
        }
      } else if constexpr (KIND == kTQ4) {
        if (nu == 2) {
          const uint8_t* const sts[2] = {st0, myring + ((it + 1) % C::NST) * C::STAGE};
          if (nvalid >= kChunk) units_tq<D, 2, false>(sts, kChunk, r, c, qb, fac, lut, S);
          else units_tq<D, 2, true>(sts, nvalid, r, c, qb, fac, lut, S);
        } else {
          const uint8_t* const sts[1] = {st0};
          if (nvalid >= kChunk) units_tq<D, 1, false>(sts, kChunk, r, c, qb, fac, lut, S);
          else units_tq<D, 1, true>(sts, nvalid, r, c, qb, fac, lut, S);
        }
      } else {
        if (nvalid >= kChunk) unit_anchor<KIND, D, false>(st0, kChunk, r, c, qb, fac, S);
        else unit_anchor<KIND, D, true>(st0, nvalid, r, c, qb, fac, S);
      }
      __syncwarp();
      for (int k = 0; k < nu; ++k) {
        const int nx = i + k + C::NST;  // warp-uniform
        if (nx < nw) {
          if ((nx & 31) == 0) {
            pf = pf_next;
            pf_next = page_of_lane(nx + 32 + lane);
          }
          const int page = __shfl_sync(kFull, pf, nx & 31);
          if (!packed4(KIND)) fence_proxy_async();  // the bulk copies are async-proxy writes
          issue(nx, (it + k) % C::NST, page);
        }
      }
      i += nu;
      it += nu;
    }

    // ---------------------------------------------- combine the 4 warps
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      S.L0 += __shfl_xor_sync(kFull, S.L0, o);
      S.L1 += __shfl_xor_sync(kFull, S.L1, o);
    }
    if (packed4(KIND) && __any_sync(kFull, S.bad != 0)) S.L0 = S.L1 = __int_as_float(0x7FC00000);
    if (r == 0) {
      comb_ml[(warp * kHB + 2 * c) * 2] = S.M0;
      comb_ml[(warp * kHB + 2 * c) * 2 + 1] = S.L0;
      comb_ml[(warp * kHB + 2 * c + 1) * 2] = S.M1;
      comb_ml[(warp * kHB + 2 * c + 1) * 2 + 1] = S.L1;
    }
    // FP4: P.V ran on values * 2^(127 - RV); TQ4: on norms * 2^(126 - RV)
    const float osc = KIND == kFP4   ? pow2i(static_cast<int>(S.RV) - 127)
                      : KIND == kTQ4 ? pow2i(static_cast<int>(S.RV) - 126)
                                     : (KIND == kFP8 ? p.v_scale : 1.f);
    {
      float* co = comb_o + warp * kHB * D;
#pragma unroll
      for (int m = 0; m < C::NMMA; ++m) {
        const int ch0 = r * C::VPT + 2 * m, ch1 = ch0 + 1;
        co[(2 * c) * D + ch0] = S.O[m][0] * osc;
        co[(2 * c + 1) * D + ch0] = S.O[m][1] * osc;
        co[(2 * c) * D + ch1] = S.O[m][2] * osc;
        co[(2 * c + 1) * D + ch1] = S.O[m][3] * osc;
      }
    }
    __syncthreads();
    {
      const int h = tid >> 4;  // 8 heads x 16 threads
      constexpr int PER = D / 16;
      const int ch = (tid & 15) * PER;
      float Ms = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) Ms = fmaxf(Ms, comb_ml[(w * kHB + h) * 2]);
      float wt[kWarps], Ls = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        wt[w] = ex2(comb_ml[(w * kHB + h) * 2] - Ms);
        Ls += wt[w] * comb_ml[(w * kHB + h) * 2 + 1];
      }
      const int64_t slot_id = static_cast<int64_t>(blockIdx.x) + pair;
      float* dst = p.ws_o + (slot_id * kHB + h) * D + ch;
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) acc += wt[w] * comb_o[(w * kHB + h) * D + ch + e];
        dst[e] = acc;
      }
      if ((tid & 15) == 0) {
        p.ws_ml[(slot_id * kHB + h) * 2] = Ms;
        p.ws_ml[(slot_id * kHB + h) * 2 + 1] = Ls;
      }
      if (tid == 0) {
        const uint32_t tag = (p.epoch << kCtaBits) | blockIdx.x;
        if (j0 == 0) p.ws_info[2 * pair] = tag;
        if (j0 + seg == nb) p.ws_info[2 * pair + 1] = tag;
      }
    }
    __syncthreads();
    if (abort_flag) break;
    u += seg;
  }
  pdl_trigger();  // the merge may now be scheduled; it still waits for the whole grid
}

// N consecutive floats, aligned for one vector load.
template <int N>
struct alignas(4 * N) VecF {
  float x[N];
};

// Log-sum-exp merge of the partials of each (sequence, query head), then the
// inverse rotation (FP4).  One warp per output row.
struct MergeParams {
  const float* ws_o;
  const float* ws_ml;
  const uint32_t* ws_info;
  uint32_t epoch;
  const int64_t* ws_units;
  const int32_t* seq_lens;
  int B, Hq, Hkv, G, nhb, cap, num_ctas;
  float* out;
  unsigned int* status;
  uqh::SignMasks sign;
  // Cascade (casc_cu == nullptr: none): the shared-prefix partials of each
  // group's sequences, [items][px_rows] (m, l) and O, merged in as well.
  const int32_t* casc_cu;
  const int32_t* casc_prefix;
  int casc_groups, casc_min_rows, casc_cap;
  const float* px_ml;
  const float* px_o;
  const int32_t* px_item_pre;
  int px_splits, px_rows;
  int64_t px_max_items;
};

template <int KIND, int D>
__global__ void __launch_bounds__(128) merge_kernel(const __grid_constant__ MergeParams p) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  pdl_wait();  // the partials come from the decode kernel
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (row >= static_cast<int64_t>(p.B) * p.Hq) return;
  const int b = static_cast<int>(row / p.Hq), h = static_cast<int>(row - static_cast<int64_t>(b) * p.Hq);
  int L = p.seq_lens[b];
  L = L < 0 ? 0 : (L > p.cap ? p.cap : L);
  float o[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) o[e] = 0.f;
  // cascade: the keys the shared-prefix kernel took, and where its partials of this row are
  const int skip = casc_skip(p, b);
  const bool dec = L > skip;  // the decode took keys skip .. L - 1
  int64_t pitem = -1;
  int prr = 0;
  if (skip > 0 && p.px_item_pre[p.casc_groups] <= p.px_max_items) {
    const int g = casc_group(p.casc_cu, p.casc_groups, b);
    const int n = p.casc_cu[g + 1] - p.casc_cu[g], i = b - p.casc_cu[g];
    const int kvh = h / p.G, rowi = i * p.G + (h - kvh * p.G), rt = rowi / p.px_rows;
    prr = rowi - rt * p.px_rows;
    pitem = p.px_item_pre[g] + (static_cast<int64_t>(kvh) * ((n * p.G + p.px_rows - 1) / p.px_rows) + rt) * p.px_splits;
  }
  if (dec || pitem >= 0) {
    const int kvh = h / p.G, hl = h - kvh * p.G, hb = hl / kHB, hh = hl - hb * kHB;
    const int pair = (b * p.Hkv + kvh) * p.nhb + hb;
    int first = 1, last = 0;
    if (dec) {
      // Entries carry this call's epoch; anything else was left by an earlier
      // call, i.e. no block of this call wrote the entry (one gave up).
      const uint32_t e0 = p.ws_info[2 * pair], e1 = p.ws_info[2 * pair + 1];
      first = static_cast<int>(e0 & kCtaMask);
      last = static_cast<int>(e1 & kCtaMask);
      if ((e0 >> kCtaBits) != p.epoch || (e1 >> kCtaBits) != p.epoch || last < first || last >= p.num_ctas) {
        record_error(p.status, kErrTimeout);
        first = 1;
        last = 0;
      }
    }
    const int64_t U = *p.ws_units;
    float Ms = -INFINITY, Ls = 0.f;
    if (pitem < 0 && last >= first && last - first < 8) {
      // Up to 8 partials (the usual case): one round of loads -- lane j's (m, l) of
      // slot first + j and every lane's channels of all the slots' O rows -- then
      // the same weights and the same slot-order sums as the general path below.
      const int s = first + lane;
      int64_t lo = 0, hi = 0;
      if (s <= last) block_range(s, U, p.num_ctas, lo, hi);
      const unsigned valid = __ballot_sync(kFull, lo < hi);
      float m = -INFINITY, lv = 0.f;
      if (lo < hi) {
        const int64_t id = (int64_t)(s + pair) * kHB + hh;
        m = p.ws_ml[id * 2];
        lv = p.ws_ml[id * 2 + 1];
      }
      VecF<EPL> v[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if ((valid >> t) & 1u)
          v[t] = *reinterpret_cast<const VecF<EPL>*>(p.ws_o + ((int64_t)(first + t + pair) * kHB + hh) * D + lane * EPL);
        else
          v[t] = VecF<EPL>{};
      }
      Ms = m;
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) Ms = fmaxf(Ms, __shfl_xor_sync(kFull, Ms, k));
      const float w = (lo < hi) ? ex2(m - Ms) : 0.f;
      Ls = w * lv;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const float wt = __shfl_sync(kFull, w, t);
        if ((valid >> t) & 1u)
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[e] += wt * v[t].x[e];
      }
    } else {
      // The partials of this row are slots first..last (those with an empty
      // unit range wrote nothing).  Their (m, l) are read lane-parallel, 32 at a
      // time; the O rows are then summed in slot order, four loads in flight.
      for (int base = first; base <= last; base += 32) {
        const int s = base + lane;
        int64_t lo = 0, hi = 0;
        if (s <= last) block_range(s, U, p.num_ctas, lo, hi);
        if (lo < hi) Ms = fmaxf(Ms, p.ws_ml[((int64_t)(s + pair) * kHB + hh) * 2]);
      }
      // The decode's partials carry p * 2^kPShift against their maximum, the shared-prefix
      // kernel's plain p: its maxima enter the merge raised by kPShift.
      if (pitem >= 0)
        for (int s = lane; s < p.px_splits; s += 32)
          Ms = fmaxf(Ms, p.px_ml[((pitem + s) * p.px_rows + prr) * 2] + kPShift);
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) Ms = fmaxf(Ms, __shfl_xor_sync(kFull, Ms, k));
      for (int base = first; base <= last; base += 32) {
        const int s = base + lane;
        int64_t lo = 0, hi = 0;
        if (s <= last) block_range(s, U, p.num_ctas, lo, hi);
        float w = 0.f;
        if (lo < hi) {
          const int64_t id = (int64_t)(s + pair) * kHB + hh;
          w = ex2(p.ws_ml[id * 2] - Ms);
          Ls += w * p.ws_ml[id * 2 + 1];
        }
        const unsigned valid = __ballot_sync(kFull, lo < hi);
        const int n = last - base + 1 < 32 ? last - base + 1 : 32;
        int j = 0;
        for (; j + 4 <= n; j += 4) {
          VecF<EPL> v[4];
          float wj[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            wj[t] = __shfl_sync(kFull, w, j + t);
            if ((valid >> (j + t)) & 1u)
              v[t] = *reinterpret_cast<const VecF<EPL>*>(p.ws_o + ((int64_t)(base + j + t + pair) * kHB + hh) * D + lane * EPL);
            else
              v[t] = VecF<EPL>{};
          }
#pragma unroll
          for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[e] += wj[t] * v[t].x[e];
        }
        for (; j < n; ++j) {
          const float wj = __shfl_sync(kFull, w, j);
          if ((valid >> j) & 1u) {
            const VecF<EPL> v = *reinterpret_cast<const VecF<EPL>*>(p.ws_o + ((int64_t)(base + j + pair) * kHB + hh) * D + lane * EPL);
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[e] += wj * v.x[e];
          }
        }
      }
      if (pitem >= 0) {  // the shared-prefix splits; an empty split (m = -inf) wrote no O row
        for (int s0 = 0; s0 < p.px_splits; s0 += 32) {
          const int s = s0 + lane;
          float w = 0.f;
          bool live = false;
          if (s < p.px_splits) {
            const float m = p.px_ml[((pitem + s) * p.px_rows + prr) * 2] + kPShift;
            live = m != -INFINITY;
            if (live) {
              w = ex2(m - Ms);
              Ls += w * p.px_ml[((pitem + s) * p.px_rows + prr) * 2 + 1];
            }
          }
          const unsigned mask = __ballot_sync(kFull, live);
          const int cnt = min(32, p.px_splits - s0);
          int j = 0;
          for (; j + 8 <= cnt; j += 8) {  // eight O rows in flight, summed in split order
            VecF<EPL> v[8];
            float wj[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              wj[t] = __shfl_sync(kFull, w, j + t);
              if ((mask >> (j + t)) & 1u)
                v[t] = *reinterpret_cast<const VecF<EPL>*>(p.px_o + ((pitem + s0 + j + t) * p.px_rows + prr) * D +
                                                           lane * EPL);
              else
                v[t] = VecF<EPL>{};
            }
#pragma unroll
            for (int t = 0; t < 8; ++t)
#pragma unroll
              for (int e = 0; e < EPL; ++e) o[e] += wj[t] * v[t].x[e];
          }
          for (; j < cnt; ++j) {
            const float wj = __shfl_sync(kFull, w, j);
            if ((mask >> j) & 1u) {
              const VecF<EPL> v =
                  *reinterpret_cast<const VecF<EPL>*>(p.px_o + ((pitem + s0 + j) * p.px_rows + prr) * D + lane * EPL);
#pragma unroll
              for (int e = 0; e < EPL; ++e) o[e] += wj * v.x[e];
            }
          }
        }
      }
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) Ls += __shfl_xor_sync(kFull, Ls, k);
    const float inv = 1.f / Ls;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] *= inv;
    if (packed4(KIND)) inverse_rotate_warp<D>(o, lane, p.sign.m);  // out = R^T o
  }
  float* dst = p.out + row * D + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; ++e) dst[e] = o[e];
  pdl_trigger();
}

// The rotated E4M3 query of n rows (the decode prologue on its own), for the
// chunked-prefill and cascade paths and the query stage hook.  One warp
// handles 8 query rows.
template <int D>
__global__ void query_fp8_kernel(const uint16_t* q, int64_t n, uint8_t* out,
                                  const __grid_constant__ uqh::SignMasks sm) {
  const int lane = threadIdx.x & 31, r = lane >> 2, c = lane & 3;
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 8 + r;
  const bool valid = row < n;
  uint32_t bytes[D / 16];
  rotated_query_bytes<D>(q + (valid ? row : 0) * D, valid, c, sm, bytes);
  if (valid)
    for (int e = 0; e < D / 16; ++e)
      *reinterpret_cast<uint32_t*>(out + row * D + c * (D / 4) + 4 * e) = bytes[e];
}

// Stage hook: the merge's inverse rotation alone, one fp32 row per warp.
template <int D>
__global__ void inverse_rotate_kernel(const float* x, int64_t n, float* y, const __grid_constant__ uqh::SignMasks sm) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= n) return;  // warp-uniform
  float o[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) o[e] = x[row * D + lane * EPL + e];
  inverse_rotate_warp<D>(o, lane, sm.m);
#pragma unroll
  for (int e = 0; e < EPL; ++e) y[row * D + lane * EPL + e] = o[e];
}

// ------------------------------------------------------------------ host
size_t ws_slot_bytes(int d) { return static_cast<size_t>(kHB) * (d + 2) * sizeof(float); }
// Workspace: [256-byte header: unit count][pair info, 2 x int32][per-slot (m, l) x 8 heads][per-slot O x 8 heads]
size_t ws_info_bytes(int64_t pairs) { return 256 + (((static_cast<size_t>(pairs) * 2 * sizeof(int32_t)) + 255) & ~size_t(255)); }

template <int KIND, int D>
uq_status run_decode(const uqh::DecodeArgs& a, int nhb, cudaStream_t s) {
  using C = DC<KIND, D>;
  const uq_cache& c = *a.cache;
  const int G = a.num_q_heads / c.num_kv_heads;
  const int pairs = a.batch * c.num_kv_heads * nhb;
  const size_t smem = C::smem_fixed + (static_cast<size_t>(a.batch) + 1) * sizeof(int);
  // the FP4 / TQ4 copy path indexes physical rows (page * Hkv + head) * page_size + offset in 32 bits
  if (packed4(KIND) && static_cast<uint64_t>(c.num_pages) * c.num_kv_heads * c.page_size > 0xFFFFFFFFull)
    return UQ_ERR_UNSUPPORTED;
  auto kern = decode_kernel<KIND, D>;
  const uqh::DevInfo& di = uqh::dev_info();
  // FP4 at head_dim 128: the tensor-memory kernel (one CTA per SM)
  const bool tc = KIND == kFP4 && D == 128 && c.page_size >= kChunk && uqdec::decode_tc_enabled() &&
                  uqdec::decode_tc_smem(a.batch) <= di.smem_optin;
  if (smem > di.smem_optin) return UQ_ERR_UNSUPPORTED;
  // The shared-memory attribute is per device and kernel; it is raised to the
  // largest size seen so far on each device (host threads may call concurrently).
  static std::mutex cfg_mu;
  static size_t cfg_smem[uqh::kMaxDevices];
  static int cfg_per_sm[uqh::kMaxDevices];
  if (di.device < 0) return UQ_ERR_CUDA;
  int per_sm;
  {
    std::lock_guard<std::mutex> lk(cfg_mu);
    if (smem > cfg_smem[di.device]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return UQ_ERR_CUDA;
      // occupancy is set by registers and the fixed part of shared memory
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, C::smem_fixed) != cudaSuccess || n < 1)
        return UQ_ERR_CUDA;
      cfg_per_sm[di.device] = n;
      cfg_smem[di.device] = smem;
    }
    per_sm = cfg_per_sm[di.device];
  }
  if (tc) per_sm = 1;
  // Workspace: [pair info][per-slot (m, l) x 8 heads][per-slot O x 8 heads]
  const size_t info = ws_info_bytes(pairs);
  if (a.ws_bytes < info) return UQ_ERR_WORKSPACE;
  const int64_t fit = static_cast<int64_t>((a.ws_bytes - info) / ws_slot_bytes(D)) - pairs;
  // At least kMinUnitsPerBlock of the batch's largest possible number of
  // 16-token units per block: every block's partial is one more step of the
  // merge, which for a small batch costs more than the parallelism gains.
  constexpr int64_t kMinUnitsPerBlock = 4;
  const int64_t max_units =
      static_cast<int64_t>(a.batch) * ((static_cast<int64_t>(a.max_pages) * c.page_size + kChunk - 1) / kChunk) *
      c.num_kv_heads * nhb;
  int64_t grid = std::min<int64_t>(static_cast<int64_t>(di.sms) * per_sm, fit);
  grid = std::min<int64_t>(grid, std::max<int64_t>(1, max_units / kMinUnitsPerBlock));
  if (grid < 1) return UQ_ERR_WORKSPACE;
  grid = std::min<int64_t>(grid, kCtaMask + 1);  // block indices fit the pair entries
  const int64_t slots = grid + pairs;
  DecParams p;
  uqh::take_decode_stall(&p.stall_cta, &p.stall_budget);
  p.q = static_cast<const uint16_t*>(a.q);
  p.kc = static_cast<const uint8_t*>(c.k_codes);
  p.ks = static_cast<const uint8_t*>(c.k_scales);
  p.vc = static_cast<const uint8_t*>(c.v_codes);
  p.vs = static_cast<const uint8_t*>(c.v_scales);
  p.k_scale = c.k_scale;
  p.v_scale = c.v_scale;
  p.block_table = a.block_table;
  p.max_pages = a.max_pages;
  p.seq_lens = a.seq_lens;
  p.B = a.batch;
  p.Hq = a.num_q_heads;
  p.Hkv = c.num_kv_heads;
  p.G = G;
  p.nhb = nhb;
  p.ps_log2 = uqh::ilog2(c.page_size);
  p.num_pages = c.num_pages;
  const float sm = a.sm_scale > 0.f ? a.sm_scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  p.sl2e = sm * 1.4426950408889634f;
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  p.ws_units = reinterpret_cast<int64_t*>(ws);
  p.ws_info = reinterpret_cast<uint32_t*>(ws + 256);
  static std::atomic<uint32_t> epoch_counter{0};
  p.epoch = epoch_counter.fetch_add(1, std::memory_order_relaxed) & kEpochMask;
  p.ws_ml = reinterpret_cast<float*>(ws + info);
  p.ws_o = p.ws_ml + slots * kHB * 2;
  p.status = uqh::status_word();
  if (!p.status) return UQ_ERR_CUDA;
  if (packed4(KIND)) uqh::make_sign_masks(c.rot_seed, D, &p.sign);
  for (int i = 0; i < 4; ++i) p.tq_lut[i] = 0;
  if (KIND == kTQ4) {
    uqh::TqTables tt;
    const uq_status st = uqh::tq_tables(D, &tt);
    if (st != UQ_OK) return st;
    for (int i = 0; i < 4; ++i) p.tq_lut[i] = tt.lut[i];
  }
  p.k_new = a.k_new;
  p.v_new = a.v_new;
  p.new_slots = a.new_slots;
  p.new_f32 = a.new_f32;
  p.num_slots = static_cast<int64_t>(c.num_pages) * c.page_size;
  p.wkc = static_cast<uint8_t*>(c.k_codes);
  p.wks = static_cast<uint8_t*>(c.k_scales);
  p.wvc = static_cast<uint8_t*>(c.v_codes);
  p.wvs = static_cast<uint8_t*>(c.v_scales);
  p.fp4_c = uqh::fp4_c(c);
  p.casc_cu = a.casc.cu;
  p.casc_prefix = a.casc.prefix;
  p.casc_groups = a.casc.groups;
  p.casc_min_rows = a.casc.min_rows;
  p.casc_cap = a.casc.cap;
  if constexpr (KIND == kFP4 && D == 128) {
    if (tc) {
      if (p.new_slots != nullptr) {
        if (uqh::launch_pdl(append_step_kernel<D>, (unsigned)(a.batch * c.num_kv_heads), 32, 0, s, p) !=
            cudaSuccess)
          return UQ_ERR_CUDA;
        p.new_slots = nullptr;
      }
      const uq_status st = uqdec::launch_decode_tc(p, static_cast<int>(grid), s);
      if (st != UQ_OK) return st;
    }
  }
  if (!tc && uqh::launch_pdl(kern, (unsigned)grid, kThreads, smem, s, p) != cudaSuccess) return UQ_ERR_CUDA;

  MergeParams mp;
  mp.ws_o = p.ws_o;
  mp.ws_ml = p.ws_ml;
  mp.ws_info = p.ws_info;
  mp.epoch = p.epoch;
  mp.ws_units = p.ws_units;
  mp.seq_lens = a.seq_lens;
  mp.B = a.batch;
  mp.Hq = a.num_q_heads;
  mp.Hkv = c.num_kv_heads;
  mp.G = G;
  mp.nhb = nhb;
  mp.cap = a.max_pages * c.page_size;
  mp.num_ctas = static_cast<int>(grid);
  mp.out = a.out;
  mp.status = p.status;
  mp.sign = p.sign;
  mp.casc_cu = a.casc.cu;
  mp.casc_prefix = a.casc.prefix;
  mp.casc_groups = a.casc.groups;
  mp.casc_min_rows = a.casc.min_rows;
  mp.casc_cap = a.casc.cap;
  mp.px_ml = a.px.ml;
  mp.px_o = a.px.o;
  mp.px_item_pre = a.px.item_pre;
  mp.px_splits = a.px.splits;
  mp.px_rows = a.px.rows;
  mp.px_max_items = a.px.max_items;
  const int64_t rows = static_cast<int64_t>(a.batch) * a.num_q_heads;
  return uqh::cuda_status(uqh::launch_pdl(merge_kernel<KIND, D>, (unsigned)((rows + 3) / 4), 128, 0, s, mp));
}

}  // namespace

namespace uqh {

namespace {
std::mutex stall_mu;
int stall_cta = -1;
long long stall_budget = 0;
}  // namespace

void arm_decode_stall(int cta, long long budget) {
  std::lock_guard<std::mutex> lk(stall_mu);
  stall_cta = cta;
  stall_budget = budget;
}

void take_decode_stall(int* cta, long long* budget) {
  std::lock_guard<std::mutex> lk(stall_mu);
  *cta = stall_cta;
  *budget = stall_budget;
  stall_cta = -1;
}

int decode_max_ctas() { return dev_info().sms * 8; }

size_t decode_workspace_bytes(int batch, int hq, int hkv, int d, int max_ctas) {
  const int G = hq / hkv;
  const int nhb = (G + kHB - 1) / kHB;
  const int64_t pairs = static_cast<int64_t>(batch) * hkv * nhb;
  return ws_info_bytes(pairs) + static_cast<size_t>(max_ctas + pairs) * ws_slot_bytes(d);
}

uq_status launch_decode(const DecodeArgs& a, cudaStream_t s) {
  const uq_cache& c = *a.cache;
  const int G = a.num_q_heads / c.num_kv_heads;
  const int nhb = (G + kHB - 1) / kHB;
  const int d = c.head_dim;
  switch (c.dtype) {
    case UQ_FP4_UE8M0:
      if (d == 256) return a.new_slots ? UQ_ERR_UNSUPPORTED : run_decode<kFP4, 256>(a, nhb, s);
      return d == 128 ? run_decode<kFP4, 128>(a, nhb, s) : run_decode<kFP4, 64>(a, nhb, s);
    case UQ_FP8_E4M3:
      if (d == 256) return run_decode<kFP8, 256>(a, nhb, s);
      return d == 128 ? run_decode<kFP8, 128>(a, nhb, s) : run_decode<kFP8, 64>(a, nhb, s);
    case UQ_TQ4:
      if (d == 256) return UQ_ERR_UNSUPPORTED;
      return d == 128 ? run_decode<kTQ4, 128>(a, nhb, s) : run_decode<kTQ4, 64>(a, nhb, s);
    default:
      if (d == 256) return run_decode<kBF16, 256>(a, nhb, s);
      return d == 128 ? run_decode<kBF16, 128>(a, nhb, s) : run_decode<kBF16, 64>(a, nhb, s);
  }
}

uq_status launch_inverse_rotate(const float* x, int64_t n, int d, uint64_t seed, float* y, cudaStream_t s) {
  SignMasks sm;
  make_sign_masks(seed, d, &sm);
  const unsigned grid = (unsigned)((n + 3) / 4);
  if (d == 256)
    inverse_rotate_kernel<256><<<grid, 128, 0, s>>>(x, n, y, sm);
  else if (d == 128)
    inverse_rotate_kernel<128><<<grid, 128, 0, s>>>(x, n, y, sm);
  else
    inverse_rotate_kernel<64><<<grid, 128, 0, s>>>(x, n, y, sm);
  return cuda_status(cudaGetLastError());
}

uq_status launch_query_fp8(const void* q, int64_t n, int d, uint64_t seed, uint8_t* out, cudaStream_t s) {
  SignMasks sm;
  make_sign_masks(seed, d, &sm);
  const int64_t warps = (n + 7) / 8;
  const unsigned grid = (unsigned)((warps + 3) / 4);
  if (d == 256)
    query_fp8_kernel<256><<<grid, 128, 0, s>>>(static_cast<const uint16_t*>(q), n, out, sm);
  else if (d == 128)
    query_fp8_kernel<128><<<grid, 128, 0, s>>>(static_cast<const uint16_t*>(q), n, out, sm);
  else
    query_fp8_kernel<64><<<grid, 128, 0, s>>>(static_cast<const uint16_t*>(q), n, out, sm);
  return cuda_status(cudaGetLastError());
}

}  // namespace uqh
