// uq_decode_tc.cu -- FP4 decode attention on the fifth-generation tensor
// cores (tcgen05, tensor memory), head_dim 128.
//
// Same arithmetic as the warp-level decode in uq_decode.cu ("UltraQuant: 4-bit
// KV Caching for Context-Heavy Agents", review, manon006.tistory.com/395,
// §3.2 and §4.2): the query is rotated and rounded to E4M3 once, keys and
// values stay E2M1 codes with UE8M0 group scales, P.V is summed per tile in a
// fresh accumulator and added to the running output in fp32, the output is
// rotated back by the merge.  Same work split (16-token units of (sequence,
// kv head, head block) cut into equal contiguous ranges, one per CTA), same
// partial layout, same merge.
//
// GB300 design: one CTA per SM takes its units in tiles of 128 tokens (8
// units) and runs each tile through a warp-specialised pipeline:
//   * warp 8 copies the tile's K codes, V codes and both scale rows (136 bytes
//     per token) into a ring of raw stages: the code rows of each unit (1 KB,
//     contiguous in a page) by bulk copies on the TMA engine, the scale rows
//     by per-lane 16-byte cp.async, all completing the stage's mbarrier; page
//     numbers are loaded two tiles ahead.
//   * warps 0-3 (thread t = token row t of the tile): repack the K row into
//     the padded E2M1 operand (16 codes in the first 8 bytes of every 16-byte
//     chunk, 128-byte swizzle) and write the row's four scale bytes to tensor
//     memory as the A scale factors; then, once QK^T is done, read the row's
//     logits from tensor memory and run the online softmax (running maximum
//     raised lazily, shared by the four warps), writing P as hi + lo f16
//     parts into shared memory.
//   * warp 9 (one thread) issues QK^T as block-scaled MMAs (kind::mxf8f6f4,
//     A = the 128 K rows in E2M1 with their UE8M0 bytes, B = the 8 query
//     heads in E4M3 with scale 1, one MMA per 32-channel group: the group
//     scale is exactly the MX block scale) and P.V as kind::f16 MMAs
//     (A = V' MN-major, B = P), both into tensor memory.
//   * warps 4-7 (thread t = token row t): convert the V row to
//     V' = code * 2^(byte - RV) in f16 (RV = the tile's largest V scale byte,
//     so the multipliers are <= 1), MN-major for the P.V MMA; then fold the
//     tile's O^T (lane = channel) into the running fp32 output in registers,
//     rescaled for a grown maximum, and at the end of a segment write the
//     partial (m, l, O) for the merge.
// Buffers between the stages are double-buffered (S, O^T, K operand, scale
// factors, V', P) so that QK^T of tile i+1 and the conversion of tile i+1
// overlap the softmax and P.V of tile i.  Every wait is bounded: on timeout
// the kernel records the error and stops waiting (all roles keep the same
// control flow, so the named barriers still match) and winds down.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "uq_decode_common.cuh"
#include "uq_device.cuh"
#include "uq_internal.h"
#include "uq_tc.cuh"

namespace {

using namespace uqd;
using namespace uqdec;
using namespace uqtc;

constexpr int kD = 128;
constexpr int kTok = 128;                   // tokens per tile
constexpr int kTUnits = kTok / kChunk;      // units per tile
constexpr int kNst = 4;                     // raw stages
constexpr int kTcThreads = 320;             // warps 0-3 softmax, 4-7 convert, 8 copy, 9 MMA
constexpr int kRowK = kD / 2;               // code bytes per token row
constexpr int kRowS = kD / 32;              // scale bytes per token row
// raw stage: [128][64] K codes, [128][64] V codes, [128][4] K scales, [128][4] V scales
constexpr int kRawV = kTok * kRowK;
constexpr int kRawKS = 2 * kTok * kRowK;
constexpr int kRawVS = kRawKS + kTok * kRowS;
constexpr int kRaw = kRawVS + kTok * kRowS;
// operands (1024-byte aligned)
constexpr int kOffK = 0;                        // [2][128 rows][128 B] padded E2M1 K, 128-byte swizzle
constexpr int kOffV = kOffK + 2 * kTok * 128;   // [2][2 halves][128 tokens][128 B] V' f16, MN-major
constexpr int kVHalf = kTok * 128;
constexpr int kOffP = kOffV + 2 * 2 * kVHalf;   // [2][hi, lo][2 atoms][16 heads][128 B] P f16, K-major
constexpr int kPPart = 2 * 16 * 128;
constexpr int kOffQ = kOffP + 2 * 2 * kPPart;   // [2][16 heads][128 B] E4M3 query, K-major
constexpr int kOffRaw = kOffQ + 2 * 16 * 128;
constexpr int kOffMisc = kOffRaw + kNst * kRaw;
constexpr int kMisc = 2048;
constexpr int kOffPre = kOffMisc + kMisc;
constexpr size_t kSmemFixed = kOffPre + 1024;  // + the 1024-byte alignment slack
// tensor-memory columns (32-column aligned)
constexpr uint32_t kColS = 0;      // S[2]: 16 columns each (8 heads used)
constexpr uint32_t kColO = 64;     // O^T[2]
constexpr uint32_t kColSfa = 128;  // K scale factors [2], 4 columns each
constexpr uint32_t kColSfb = 192;  // query scale factors (all 1)
constexpr int kTmemCols = 256;

// barriers in the misc area
enum Bar {
  kBarFull = 0,                  // [kNst] raw stage landed (32 copy lanes)
  kBarEmpty = kBarFull + kNst,   // [kNst] raw stage read (8 warps)
  kBarKReady = kBarEmpty + kNst, // [2] K operand + scale factors written (4 softmax warps)
  kBarSFull = kBarKReady + 2,    // [2] QK^T done (MMA commit)
  kBarPReady = kBarSFull + 2,    // [2] P written, S read (4 softmax warps)
  kBarVReady = kBarPReady + 2,   // [2] V' written (4 convert warps)
  kBarOFull = kBarVReady + 2,    // [2] P.V done (MMA commit)
  kBarOFree = kBarOFull + 2,     // [2] O^T read (4 convert warps)
  kBarDone = kBarOFree + 2,      // every MMA complete
  kBarCount = kBarDone + 1
};
// other misc fields (byte offsets)
constexpr int kMiscTslot = 256;
constexpr int kMiscAbort = 260;
constexpr int kMiscMref = 272;               // [4 tiles][8] float: the running maximum each tile's P used
constexpr int kMiscGflag = kMiscMref + 128;  // [2][4] int: a warp saw a logit above max + slack
constexpr int kMiscGmax = kMiscGflag + 32;   // [4][8] float: warp maxima of a tile
constexpr int kMiscRvx = kMiscGmax + 128;    // [2][4] uint: warp maxima of the V scale bytes
constexpr int kMiscLx = kMiscRvx + 32;       // [2 segments][4][8] float: warp sums of l
constexpr int kMiscMfin = kMiscLx + 256;     // [2 segments][8] float: final maximum
constexpr int kMiscBad = kMiscMfin + 64;     // [2 segments][8] uint: non-finite group seen (per warp)
static_assert(kMiscBad + 64 <= kMisc, "misc area");

// kind::mxf8f6f4 block-scaled: A E2M1 (the keys, M = 128 tokens), B E4M3 (the
// queries, N = 16 rows of which 8 are heads), both K-major, UE8M0 scales, scale
// byte g of each row's 32-bit scale word (g = the 32-channel group).
constexpr uint32_t idesc_qk(int g) {
  return (5u << 7) | (0u << 10) | ((16u >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) |
         (static_cast<uint32_t>(g) << 29) | (static_cast<uint32_t>(g) << 4);
}
// kind::f16: D f32, A (V', M = 128 channels) f16 MN-major, B (P, N = 16) f16 K-major.
constexpr uint32_t kIdescPV = (1u << 4) | (1u << 15) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void bar_named(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One poll of a barrier phase, without a suspend-time hint: the hand-offs of
// this pipeline take a few hundred cycles, and a parked thread is woken later
// than that.
__device__ __forceinline__ bool poll(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok)
               : "r"(smem_u32(bar)), "r"(parity)
               : "memory");
  return ok != 0;
}

// Bounded wait; after a timeout (here or in any other thread) it returns at
// once, so that every role runs to the end of its loop and the kernel exits.
__device__ __forceinline__ void tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        unsigned int* status) {
  if (poll(bar, parity)) return;
  const long long t0 = clock64();
  while (!*abort_flag) {
    __nanosleep(32);  // leave the issue slots to the warps that work
    if (poll(bar, parity)) return;
    if (clock64() - t0 > kWaitBudget) {
      record_error(status, kErrTimeout);
      *abort_flag = 1;
      return;
    }
  }
}

// The tiles of one CTA: its unit range [lo, hi) walked pair by pair (a pair is
// one (sequence, kv head, head block), nb units), at most 8 units per tile.
struct Tile {
  int b, pl, j, n;    // sequence, pair within the sequence, first unit within the pair, units
  bool first, last;   // first / last tile of this CTA's segment of the pair
};
struct Cursor {
  int64_t u, hi;
  int b, pl, j;
  bool fresh;
  __device__ void init(const int* pre, int B, int pps, int64_t lo, int64_t hi_) {
    u = lo;
    hi = hi_;
    fresh = true;
    b = 0;
    pl = 0;
    j = 0;
    if (u >= hi) return;
    int lb = 1, hb = B;  // first index with pre[idx] * pps > u
    while (lb < hb) {
      const int mid = (lb + hb) >> 1;
      if (static_cast<int64_t>(pre[mid]) * pps > u) hb = mid; else lb = mid + 1;
    }
    b = lb - 1;
    const int nb = pre[b + 1] - pre[b];
    const int64_t off = u - static_cast<int64_t>(pre[b]) * pps;
    pl = static_cast<int>(off / nb);
    j = static_cast<int>(off - static_cast<int64_t>(pl) * nb);
  }
  __device__ bool next(const int* pre, int B, int pps, Tile& t) {
    if (u >= hi) return false;
    const int nb = pre[b + 1] - pre[b];
    const int64_t left = hi - u;
    int n = nb - j < kTUnits ? nb - j : kTUnits;
    if (left < n) n = static_cast<int>(left);
    t.b = b;
    t.pl = pl;
    t.j = j;
    t.n = n;
    t.first = fresh || j == 0;
    t.last = j + n == nb || left == n;
    fresh = false;
    u += n;
    j += n;
    if (j == nb) {
      j = 0;
      if (++pl == pps) {
        pl = 0;
        ++b;
        while (b < B && pre[b + 1] == pre[b]) ++b;
      }
    }
    return true;
  }
};

struct SegInfo {  // per-pair values a role needs
  int b = -1, L = 0, ub = 0;
};
__device__ __forceinline__ void seg_info(const DecParams& p, int b, SegInfo& s) {
  if (s.b == b) return;
  s.b = b;
  s.L = clamp_len(p, b);
  s.ub = casc_skip(p, b) / kChunk;
}

__global__ void __launch_bounds__(kTcThreads, 1) decode_tc_kernel(const __grid_constant__ DecParams p) {
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  uint8_t* misc = sm + kOffMisc;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(misc + kMiscTslot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + kMiscAbort);
  float* mref = reinterpret_cast<float*>(misc + kMiscMref);
  int* gflag = reinterpret_cast<int*>(misc + kMiscGflag);
  float* gmax = reinterpret_cast<float*>(misc + kMiscGmax);
  uint32_t* rvx = reinterpret_cast<uint32_t*>(misc + kMiscRvx);
  float* lx = reinterpret_cast<float*>(misc + kMiscLx);
  float* mfin = reinterpret_cast<float*>(misc + kMiscMfin);
  uint32_t* badx = reinterpret_cast<uint32_t*>(misc + kMiscBad);
  int* pre = reinterpret_cast<int*>(sm + kOffPre);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    // stage full: the 32 copy lanes' cp.async arrivals and the bulk copies' byte count
    for (int i = 0; i < kBarFull + kNst; ++i) mbar_init(&bars[i], 33);
    for (int i = kBarEmpty; i < kBarEmpty + kNst; ++i) mbar_init(&bars[i], 8);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBarKReady + i], 4);
      mbar_init(&bars[kBarSFull + i], 1);
      mbar_init(&bars[kBarPReady + i], 4);
      mbar_init(&bars[kBarVReady + i], 4);
      mbar_init(&bars[kBarOFull + i], 1);
      mbar_init(&bars[kBarOFree + i], 4);
    }
    mbar_init(&bars[kBarDone], 1);
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = *tslot;
  if (warp < 4) {  // query scale factors: byte 127 (scale 1) for every query row and group
    const uint32_t one = 0x7F7F7F7Fu;
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tmem + (static_cast<uint32_t>(warp * 32) << 16) + kColSfb),
                 "r"(one) : "memory");
    tmem_wait_st();
  }
  pdl_wait();  // the cache, query and block table are written by earlier kernels
  // Prefix sums of 16-token units per sequence (as the warp-level decode).
  if (warp == 0) {
    int run = 0;
    if (lane == 0) pre[0] = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      int x = 0;
      if (b < p.B) {
        const int L = clamp_len(p, b), skip = casc_skip(p, b);
        if (skip > L) record_error(p.status, kErrBounds);
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
  tc_before();
  __syncthreads();
  tc_after();

  const int pps = p.Hkv * p.nhb;
  const int64_t U = static_cast<int64_t>(pre[p.B]) * pps;
  int64_t lo, hi;
  block_range(blockIdx.x, U, gridDim.x, lo, hi);
  if (blockIdx.x == 0 && tid == 0) *p.ws_units = U;
  const int ps_mask = (1 << p.ps_log2) - 1;

  if (warp < 4) {
    // ------------------------------------------------------------ softmax warps
    const int t = tid;  // token row of the tile
    float M[kHB], Lr[kHB];
#pragma unroll
    for (int h = 0; h < kHB; ++h) {
      M[h] = -INFINITY;
      Lr[h] = 0.f;
    }
    uint32_t bad = 0;
    Cursor cur, pc;
    cur.init(pre, p.B, pps, lo, hi);
    pc.init(pre, p.B, pps, lo, hi);
    SegInfo si, sp;
    int segq = 1, segc = 1;  // query buffer of the prep cursor's and of the current tile's segment
    const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
    // prep: the K operand and the scale factors of tile k (and the query at a segment start)
    auto prep = [&](const Tile& T, int k) -> uint32_t {
      const int stage = k % kNst;
      tc_wait(&bars[kBarFull + stage], (k / kNst) & 1, abort_flag, p.status);
      seg_info(p, T.b, sp);
      if (T.first) {
        segq ^= 1;
        if (warp == 0) {  // rotated E4M3 query of the pair's (up to) 8 heads, natural channel order
          const int kvh = T.pl / p.nhb, hblk = T.pl - kvh * p.nhb;
          const int r = lane >> 2, c = lane & 3;
          const int hloc = hblk * kHB + r;
          const bool hv = hloc < p.G;
          const uint16_t* qrow = p.q + (static_cast<int64_t>(T.b) * p.Hq + kvh * p.G + (hv ? hloc : 0)) * kD;
          uint32_t qb[kD / 16];
          rotated_query_bytes<kD>(qrow, hv, c, p.sign, qb);
          uint8_t* qd = sm + kOffQ + segq * 2048 + r * 128;
#pragma unroll
          for (int e = 0; e < kD / 16; ++e)
            *reinterpret_cast<uint32_t*>(qd + ((((2 * c + (e >> 2)) ^ r) & 7) << 4) + ((4 * e) & 15)) = qb[e];
        }
      }
      const uint8_t* raw = sm + kOffRaw + stage * kRaw;
      // K row t: cache word 4w + g holds natural word 4g + w (groups interleaved);
      // operand chunk 2g + h = natural words 4g + 2h, 4g + 2h + 1
      const uint4* kr = reinterpret_cast<const uint4*>(raw + t * kRowK);
      const uint4 c0 = kr[0], c1 = kr[1], c2 = kr[2], c3 = kr[3];
      const uint32_t wd[16] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w,
                               c2.x, c2.y, c2.z, c2.w, c3.x, c3.y, c3.z, c3.w};
      uint8_t* kd = sm + kOffK + (k & 1) * (kTok * 128) + (t >> 3) * 1024 + (t & 7) * 128;
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ch = 2 * g + h;
          *reinterpret_cast<uint4*>(kd + (((ch ^ t) & 7) << 4)) =
              make_uint4(wd[4 * (2 * h) + g], wd[4 * (2 * h + 1) + g], 0u, 0u);
        }
      // A scale factors: the word of row 32 j + lane in lane `lane` of this quarter, column j
      const uint32_t* ksw = reinterpret_cast<const uint32_t*>(raw + kRawKS);
      const uint32_t s0 = ksw[lane], s1 = ksw[32 + lane], s2 = ksw[64 + lane], s3 = ksw[96 + lane];
      asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                       tmem + lanes + kColSfa + 32u * (k & 1)),
                   "r"(s0), "r"(s1), "r"(s2), "r"(s3)
                   : "memory");
      const int tok = (sp.ub + T.j) * kChunk + t;
      const uint32_t kbad = (t < T.n * kChunk && tok < sp.L) ? has_ff(ksw[t]) : 0u;
      tmem_wait_st();
      fence_proxy_async();
      tc_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive1(&bars[kBarKReady + (k & 1)]);
        mbar_arrive1(&bars[kBarEmpty + stage]);
      }
      return kbad;
    };
    Tile T, TN;
    // Tiles i + 1 and i + 2 are prepared while tile i is in the softmax: the K
    // operand and scale-factor buffers of tile i + 2 are those of tile i, free once
    // its QK^T is done (waited for below).  kb0, kb1: non-finite K group bits of
    // tiles i and i + 1, found by their prep.
    uint32_t kb0 = 0, kb1 = 0;
    if (pc.next(pre, p.B, pps, TN)) kb0 = prep(TN, 0);
    if (pc.next(pre, p.B, pps, TN)) kb1 = prep(TN, 1);
    for (int i = 0; cur.next(pre, p.B, pps, T); ++i) {
      bad |= kb0;
      seg_info(p, T.b, si);
      if (T.first) segc ^= 1;
      // ---- softmax of tile i
      tc_wait(&bars[kBarSFull + (i & 1)], (i >> 1) & 1, abort_flag, p.status);
      tc_after();
      uint32_t sr[8];
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                   : "=r"(sr[0]), "=r"(sr[1]), "=r"(sr[2]), "=r"(sr[3]), "=r"(sr[4]), "=r"(sr[5]), "=r"(sr[6]),
                     "=r"(sr[7])
                   : "r"(tmem + lanes + kColS + 32u * (i & 1)));
      tmem_wait_ld();
      const int tok = (si.ub + T.j) * kChunk + t;
      const bool valid = t < T.n * kChunk && tok < si.L;
      float x[kHB];
      bool up = false;
#pragma unroll
      for (int h = 0; h < kHB; ++h) {
        x[h] = valid ? __uint_as_float(sr[h]) * p.sl2e : -INFINITY;
        up |= x[h] > M[h] + kSlack;
      }
      const unsigned vote = __ballot_sync(kFull, up);
      if (lane == 0) gflag[(i & 1) * 4 + warp] = vote != 0u;
      bar_named(1, 128);
      const int* gf = gflag + (i & 1) * 4;
      if (gf[0] | gf[1] | gf[2] | gf[3]) {  // rare: raise the maximum to this tile's exact one
        float m[kHB];
#pragma unroll
        for (int h = 0; h < kHB; ++h) {
          m[h] = x[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m[h] = fmaxf(m[h], __shfl_xor_sync(kFull, m[h], o));
        }
        if (lane < kHB) {
          float v = m[0];
#pragma unroll
          for (int h = 1; h < kHB; ++h) v = lane == h ? m[h] : v;
          gmax[warp * kHB + lane] = v;
        }
        bar_named(1, 128);
#pragma unroll
        for (int h = 0; h < kHB; ++h) {
          const float n = fmaxf(fmaxf(M[h], fmaxf(gmax[h], gmax[kHB + h])), fmaxf(gmax[2 * kHB + h], gmax[3 * kHB + h]));
          Lr[h] *= ex2(M[h] - n);
          M[h] = n;
        }
      }
      // P = 2^(x - M + kPShift) as hi (13 low mantissa bits cleared, exact in f16) + lo
      uint16_t ph[kHB], pl[kHB];
#pragma unroll
      for (int h = 0; h < kHB; ++h) {
        const float pv = ex2(x[h] - M[h] + kPShift);
        Lr[h] += pv;
        const float hv = __uint_as_float(__float_as_uint(pv) & 0xFFFFE000u);
        ph[h] = __half_as_ushort(__float2half_rn(hv));
        pl[h] = __half_as_ushort(__float2half_rn(pv - hv));
      }
      if (i >= 2) tc_wait(&bars[kBarOFull + (i & 1)], ((i - 2) >> 1) & 1, abort_flag, p.status);  // P.V of i-2 done
      uint8_t* pd = sm + kOffP + (i & 1) * (2 * kPPart) + (t >> 6) * 2048 + (t & 7) * 2;
#pragma unroll
      for (int h = 0; h < kHB; ++h) {
        const int off = h * 128 + (((((t & 63) >> 3) ^ h) & 7) << 4);
        *reinterpret_cast<uint16_t*>(pd + off) = ph[h];
        *reinterpret_cast<uint16_t*>(pd + kPPart + off) = pl[h];
      }
      if (t == 0)
#pragma unroll
        for (int h = 0; h < kHB; ++h) mref[(i & 3) * kHB + h] = M[h];
      fence_proxy_async();
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(&bars[kBarPReady + (i & 1)]);
      kb0 = kb1;
      kb1 = pc.next(pre, p.B, pps, TN) ? prep(TN, i + 2) : 0u;
      if (T.last) {  // end of the segment: l summed over the tile rows, handed to the convert warps
        const unsigned anybad = __ballot_sync(kFull, bad != 0);
#pragma unroll
        for (int h = 0; h < kHB; ++h) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) Lr[h] += __shfl_xor_sync(kFull, Lr[h], o);
        }
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < kHB; ++h) lx[(segc * 4 + warp) * kHB + h] = Lr[h];
          badx[segc * 8 + warp] = anybad != 0u;
          if (warp == 0)
#pragma unroll
            for (int h = 0; h < kHB; ++h) mfin[segc * kHB + h] = M[h];
        }
        bar_named(3, 256);
#pragma unroll
        for (int h = 0; h < kHB; ++h) {
          M[h] = -INFINITY;
          Lr[h] = 0.f;
        }
        bad = 0;
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ convert warps
    const int cw = warp - 4, t = cw * 32 + lane;  // token row t; tensor-memory quarter cw = channels 32 cw ..
    const uint32_t lanes = static_cast<uint32_t>(cw * 32) << 16;
    float O[kHB], Mr[kHB];
#pragma unroll
    for (int h = 0; h < kHB; ++h) {
      O[h] = 0.f;
      Mr[h] = -INFINITY;
    }
    uint32_t bad = 0, rvh[2] = {0u, 0u};  // RV of the last two tiles
    int folded = -1, segc = 1, seg_j0 = 0;
    Cursor cur;
    cur.init(pre, p.B, pps, lo, hi);
    SegInfo si;
    auto fold = [&](int k, uint32_t rv) {
      tc_wait(&bars[kBarOFull + (k & 1)], (k >> 1) & 1, abort_flag, p.status);
      tc_after();
      uint32_t o[8];
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                   : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]), "=r"(o[4]), "=r"(o[5]), "=r"(o[6]), "=r"(o[7])
                   : "r"(tmem + lanes + kColO + 32u * (k & 1)));
      tmem_wait_ld();
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(&bars[kBarOFree + (k & 1)]);
      const float osc = pow2i(static_cast<int>(rv) - 127);  // P.V ran on values * 2^(127 - RV)
      const float* mt = mref + (k & 3) * kHB;
#pragma unroll
      for (int h = 0; h < kHB; ++h) {
        const float m = mt[h];
        if (m != Mr[h]) {  // the maximum grew with this tile (warp-uniform)
          O[h] *= ex2(Mr[h] - m);
          Mr[h] = m;
        }
        O[h] = fmaf(__uint_as_float(o[h]), osc, O[h]);
      }
      folded = k;
    };
    Tile T;
    for (int i = 0; cur.next(pre, p.B, pps, T); ++i) {
      const int stage = i % kNst;
      seg_info(p, T.b, si);
      if (T.first) {
        segc ^= 1;
        seg_j0 = T.j;
      }
      tc_wait(&bars[kBarFull + stage], (i / kNst) & 1, abort_flag, p.status);
      const uint8_t* raw = sm + kOffRaw + stage * kRaw;
      const int tok = (si.ub + T.j) * kChunk + t;
      const bool valid = t < T.n * kChunk && tok < si.L;
      const uint32_t vsw = valid ? reinterpret_cast<const uint32_t*>(raw + kRawVS)[t] : 0u;
      bad |= has_ff(vsw);
      const uint32_t bm = max(max(vsw & 0xFFu, (vsw >> 8) & 0xFFu), max((vsw >> 16) & 0xFFu, vsw >> 24));
      const uint32_t wm = __reduce_max_sync(kFull, bm);
      if (lane == 0) rvx[(i & 1) * 4 + cw] = wm;
      bar_named(2, 128);
      const uint32_t* rv4 = rvx + (i & 1) * 4;
      const uint32_t rv_cur = max(max(rv4[0], rv4[1]), max(rv4[2], rv4[3]));
      // O^T of tile i - 2 (its P.V ran during the conversion of tile i - 1): folded
      // now, which also frees the V' buffer that tile i takes
      if (i >= 2 && folded < i - 2) fold(i - 2, rvh[i & 1]);
      rvh[i & 1] = rv_cur;
      const float rref = pow2i(127 - static_cast<int>(rv_cur));
      uint32_t mult[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const float f = __uint_as_float(((vsw >> (8 * g)) & 0xFFu) << 23) * rref;  // 2^(byte - RV); byte 0: 0
        mult[g] = pack_f16x2(f, f);
      }
      // V' row t: word q of the cache row = channels 8q .. 8q+7 (natural order)
      const uint4* vr = reinterpret_cast<const uint4*>(raw + kRawV + t * kRowK);
      uint8_t* vd = sm + kOffV + (i & 1) * (2 * kVHalf) + (t >> 3) * 1024 + (t & 7) * 128;
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const uint4 w4 = vr[qq];
        const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = 4 * qq + e;  // channels 8q .. 8q + 7, group q / 4
          uint32_t a[4];
          e2m1x8_to_f16x2(wv[e], a);
#pragma unroll
          for (int k = 0; k < 4; ++k) a[k] = hmul2(a[k], mult[qq]);
          *reinterpret_cast<uint4*>(vd + (q >> 3) * kVHalf + ((((q & 7) ^ t) & 7) << 4)) = make_uint4(a[0], a[1], a[2], a[3]);
        }
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive1(&bars[kBarVReady + (i & 1)]);
        mbar_arrive1(&bars[kBarEmpty + stage]);
      }
      if (T.last) {
        if (i >= 1 && folded < i - 1) fold(i - 1, rvh[(i - 1) & 1]);
        fold(i, rv_cur);
        const unsigned anybad = __ballot_sync(kFull, bad != 0);
        if (lane == 0) badx[segc * 8 + 4 + cw] = anybad != 0u;
        bar_named(3, 256);
        const int ch = cw * 32 + lane;
        const int pair = T.b * pps + T.pl;
        const int64_t slot_id = static_cast<int64_t>(blockIdx.x) + pair;
        uint32_t nb_any = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) nb_any |= badx[segc * 8 + w];
        if (!*abort_flag) {
#pragma unroll
          for (int h = 0; h < kHB; ++h) p.ws_o[(slot_id * kHB + h) * kD + ch] = O[h];
          if (cw == 0 && lane < kHB) {
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) l += lx[(segc * 4 + w) * kHB + lane];
            if (nb_any) l = __int_as_float(0x7FC00000);
            p.ws_ml[(slot_id * kHB + lane) * 2] = mfin[segc * kHB + lane];
            p.ws_ml[(slot_id * kHB + lane) * 2 + 1] = l;
          }
          if (cw == 0 && lane == 0) {
            const int nb = pre[T.b + 1] - pre[T.b];
            const uint32_t tag = (p.epoch << kCtaBits) | blockIdx.x;
            if (seg_j0 == 0) p.ws_info[2 * pair] = tag;
            if (T.j + T.n == nb) p.ws_info[2 * pair + 1] = tag;
          }
        }
#pragma unroll
        for (int h = 0; h < kHB; ++h) {
          O[h] = 0.f;
          Mr[h] = -INFINITY;
        }
        bad = 0;
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ copy warp
    Cursor cur, la;
    cur.init(pre, p.B, pps, lo, hi);
    la.init(pre, p.B, pps, lo, hi);
    SegInfo sl;
    const uint32_t raw0 = sb + kOffRaw;
    // lane u < 8 holds the page of unit u of a tile; loaded two tiles ahead and
    // checked where it is used, so the load's latency never stalls the copies
    auto pages = [&](Tile& X) {
      int page = 0;
      if (la.next(pre, p.B, pps, X)) {
        seg_info(p, X.b, sl);
        if (lane < X.n) {
          const int tok = (sl.ub + X.j + lane) * kChunk;
          page = p.block_table[static_cast<int64_t>(X.b) * p.max_pages + (tok >> p.ps_log2)];
        }
      }
      return page;
    };
    Tile X;
    int pg0 = pages(X), pg1 = pages(X);
    const uint32_t page_rows = static_cast<uint32_t>(p.Hkv) << p.ps_log2;
    SegInfo si;
    Tile T;
    for (int i = 0; cur.next(pre, p.B, pps, T); ++i) {
      const int stage = i % kNst;
      uint64_t* full = &bars[kBarFull + stage];
      if (i >= kNst) tc_wait(&bars[kBarEmpty + stage], ((i - kNst) / kNst) & 1, abort_flag, p.status);
      seg_info(p, T.b, si);
      const int kvh = T.pl / p.nhb;
      const uint32_t rowh = static_cast<uint32_t>(kvh) << p.ps_log2;
      const uint32_t dst = raw0 + stage * kRaw;
      // this lane's unit: K codes for lanes 0-7, V codes for lanes 16-23, scale chunk lane & 3 of unit lane >> 2
      int page = __shfl_sync(kFull, pg0, lane & 7);
      if (page < 0 || page >= p.num_pages) {
        if ((lane & 7) < T.n) record_error(p.status, kErrBounds);
        page = 0;
      }
      const int us = lane >> 2;  // scale rows: unit
      int spage = __shfl_sync(kFull, pg0, us & 7);
      if (spage < 0 || spage >= p.num_pages) spage = 0;
      if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(T.n) * 2 * kChunk * kRowK);
      __syncwarp();
      {
        const int u = lane & 7;
        const bool is_v = (lane & 16) != 0;
        if ((lane & 8) == 0 && u < T.n) {  // one 1 KB bulk copy per unit and array
          const int tok0 = (si.ub + T.j + u) * kChunk;
          const uint32_t row = static_cast<uint32_t>(page) * page_rows + rowh + (tok0 & ps_mask);
          const uint8_t* src = (is_v ? p.vc : p.kc) + static_cast<uint64_t>(row) * kRowK;
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                  dst + (is_v ? kRawV : 0) + u * (kChunk * kRowK)),
              "l"(src), "r"(uint32_t(kChunk * kRowK)), "r"(smem_u32(full))
              : "memory");
        }
      }
      if (us < T.n) {  // scale rows: lane l copies 16-byte chunk l & 3 of unit l >> 2, K and V
        const int c = lane & 3;
        const int tok0 = (si.ub + T.j + us) * kChunk;
        const uint32_t row = static_cast<uint32_t>(spage) * page_rows + rowh + (tok0 & ps_mask);
        const uint32_t ds = dst + kRawKS + us * (kChunk * kRowS) + 16 * c;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ds),
                     "l"(p.ks + static_cast<uint64_t>(row) * kRowS + 16 * c) : "memory");
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ds + kTok * kRowS),
                     "l"(p.vs + static_cast<uint64_t>(row) * kRowS + 16 * c) : "memory");
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(full)) : "memory");
      pg0 = pg1;
      pg1 = pages(X);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (lane == 0) {
    // ------------------------------------------------------------ MMA thread (warp 9)
    Cursor cur;
    cur.init(pre, p.B, pps, lo, hi);
    int segq = 1;
    auto pv = [&](int k) {
      tc_after();
      const uint32_t va = sb + kOffV + (k & 1) * (2 * kVHalf);
      const uint32_t pa = sb + kOffP + (k & 1) * (2 * kPPart);
      const uint32_t d = tmem + kColO + 32u * (k & 1);
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int s = 0; s < kTok / 16; ++s)
          tc_mma_ss(d, tc_desc_mn(va + 2048 * s, kVHalf), tc_desc(pa + part * kPPart + (s >> 2) * 2048 + (s & 3) * 32),
                    kIdescPV, (part | s) != 0 ? 1u : 0u);
      tc_commit(&bars[kBarOFull + (k & 1)]);
    };
    // Event loop: QK^T of tile nq as soon as its operands are ready (and the S
    // buffer it overwrites has been read, i.e. P.V of nq - 2 was issued), P.V of
    // tile np as soon as its P and V' are ready and its O^T buffer is free.
    Tile T;
    bool more = cur.next(pre, p.B, pps, T);
    int nq = 0, np = 0;
    long long t0 = clock64();
    while (more || np < nq) {
      bool progress = false;
      if (more && nq <= np + 1 && poll(&bars[kBarKReady + (nq & 1)], (nq >> 1) & 1)) {
        if (T.first) segq ^= 1;
        tc_after();
        const uint32_t ka = sb + kOffK + (nq & 1) * (kTok * 128);
        const uint32_t qa = sb + kOffQ + segq * 2048;
#pragma unroll
        for (int g = 0; g < 4; ++g)
          tc_mma_bs(tmem + kColS + 32u * (nq & 1), tc_desc(ka + 32 * g), tc_desc(qa + 32 * g), idesc_qk(g),
                    tmem + kColSfa + 32u * (nq & 1), tmem + kColSfb, g > 0 ? 1u : 0u);
        tc_commit(&bars[kBarSFull + (nq & 1)]);
        ++nq;
        more = cur.next(pre, p.B, pps, T);
        progress = true;
      }
      if (np < nq && poll(&bars[kBarPReady + (np & 1)], (np >> 1) & 1) &&
          poll(&bars[kBarVReady + (np & 1)], (np >> 1) & 1) &&
          (np < 2 || poll(&bars[kBarOFree + (np & 1)], ((np - 2) >> 1) & 1))) {
        pv(np);
        ++np;
        progress = true;
      }
      if (progress) {
        t0 = clock64();
      } else if (__nanosleep(32), *abort_flag) {
        break;
      } else if (clock64() - t0 > kWaitBudget) {
        record_error(p.status, kErrTimeout);
        *abort_flag = 1;
        break;
      }
    }
    tc_commit(&bars[kBarDone]);
    // the MMAs in flight finish before the tensor memory is freed, after an
    // abort too (bounded, whatever the abort flag says)
    if (!mbar_wait_sleep(&bars[kBarDone], 0, kWaitBudget)) record_error(p.status, kErrTimeout);
  }
  tc_before();
  __syncthreads();
  tc_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  pdl_trigger();
}

}  // namespace

namespace uqdec {

// Opt-in (UQ_FP4_DECODE=tc, read once per process).  The warp-level kernel
// is faster on GB300 and stays the default: 8 sequences x 64K tokens take
// 0.39 ms here against 0.14 ms there.  One copy warp per SM streams at most
// ~2 TB/s (measured with the compute roles switched off), and with only 16
// MMA columns every P.V MMA re-reads the f16 V' tile from shared memory
// (twice, for the hi and lo parts of P): ~100 KB of shared-memory traffic per
// 128-token tile on top of the copies.
bool decode_tc_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("UQ_FP4_DECODE");
    return e != nullptr && std::strcmp(e, "tc") == 0;
  }();
  return on;
}

size_t decode_tc_smem(int batch) { return kSmemFixed + (static_cast<size_t>(batch) + 1) * sizeof(int); }

uq_status launch_decode_tc(const DecParams& p, int grid, cudaStream_t s) {
  const uqh::DevInfo& di = uqh::dev_info();
  if (di.device < 0) return UQ_ERR_CUDA;
  const size_t smem = decode_tc_smem(p.B);
  if (smem > di.smem_optin) return UQ_ERR_UNSUPPORTED;
  static std::mutex mu;
  static size_t cfg[uqh::kMaxDevices];
  {
    std::lock_guard<std::mutex> lk(mu);
    if (smem > cfg[di.device]) {
      if (cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return UQ_ERR_CUDA;
      cfg[di.device] = smem;
    }
  }
  return uqh::cuda_status(uqh::launch_pdl(decode_tc_kernel, (unsigned)grid, kTcThreads, smem, s, p));
}

}  // namespace uqdec
