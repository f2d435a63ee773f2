// uq_prefill.cu -- chunked-prefill attention over the FP4 cache.
//
// A prefill chunk appends n_b new tokens to sequence b (quantize-append, as in
// the decode path) and then lets every new token attend, causally, to all of
// the sequence's tokens in the cache: query i of the chunk sits at position
// p = seq_len_b - n_b + i and sees keys 0..p.  The numerics are the decode's
// ("UltraQuant" review, manon006.tistory.com/395, §3.2): the query is rotated
// and rounded to E4M3, keys and values are E2M1 codes with UE8M0 group scales,
// the output is rotated back.
//
// GB300 design (many query rows per key: a dense contraction, unlike decode)
//   * A block takes 64 query rows of one (sequence, kv head) -- consecutive
//     (token, head) pairs of the chunk, 16 per warp -- and one range of keys.
//     Keys arrive in tiles of 64 tokens: the page rows of the tile's K codes,
//     V codes and both scale rows come by 1-D bulk copies (TMA engine) into a
//     ring of raw stages; the block converts each tile ONCE into f16 tiles in
//     shared memory (K: the codes, exact; V: code * 2^(byte - RV), RV the
//     block's running maximum V scale byte), so the conversion is shared by
//     the 64 query rows instead of being repeated per 8 heads as in decode.
//   * Each warp runs FlashAttention-style m16n8k16 MMAs: QK^T with B from
//     ldmatrix on the swizzled K tile, one 32-channel group at a time into a
//     fresh accumulator, times the group's 2^(byte-127) in fp32; online
//     softmax on the register fragments; P (hi + lo f16 parts) as the A operand
//     straight from the S fragments; P.V with B from ldmatrix.trans on the V
//     tile, each tile summed in a fresh accumulator and added to the fp32
//     output with IEEE rounding (as in decode).
//   * Long key ranges are split over blocks; each (row tile, key split) writes
//     a partial (m, l, O) and a merge kernel combines them by log-sum-exp and
//     applies the inverse rotation.
#include <algorithm>
#include <cmath>

#include "uq_device.cuh"
#include "uq_internal.h"

namespace {

using namespace uqd;

constexpr int kPWarps = 4;
constexpr int kPThreads = 32 * kPWarps;
constexpr int kPRows = 16 * kPWarps;  // query rows per block
constexpr int kKT = 64;               // keys per tile
constexpr int kPNST = 3;              // raw stages in the ring

template <int D>
struct PC {
  static constexpr int KROW = D / 2;             // code bytes per row
  static constexpr int SROW = D / 32;            // scale bytes per row
  static constexpr int NG = D / 32;              // groups
  static constexpr int RAW = 2 * kKT * KROW + 2 * kKT * SROW;  // one raw tile
  static constexpr int TILEB = kKT * D * 2;      // one f16 tile (K or V)
  static constexpr int QB = 16 * D;              // E4M3 query bytes per warp
  // raw ring | K f16 | V f16 | K scales (fp32 [NG][kKT]) | query staging | barriers + block state
  static constexpr int OFF_K = kPNST * RAW;
  static constexpr int OFF_V = OFF_K + TILEB;
  static constexpr int OFF_S = OFF_V + TILEB;
  static constexpr int OFF_Q = OFF_S + NG * kKT * 4;
  static constexpr int OFF_B = OFF_Q + kPWarps * QB;
  static constexpr int SMEM = OFF_B + 128;
};

struct PrefillParams {
  const uint8_t* qbytes;     // rotated E4M3 query, [T][Hq][D]
  const int32_t* cu_q;       // [B + 1] first query token of each sequence
  const int32_t* seq_lens;   // [B] keys of each sequence after the chunk
  const int32_t* block_table;
  int max_pages;
  const uint8_t* kc;
  const uint8_t* ks;
  const uint8_t* vc;
  const uint8_t* vs;
  int B, T, Hq, Hkv, G, ps_log2, num_pages;
  int splits;                // key splits per row tile
  int kchunk;                // keys per split (multiple of kKT)
  float sl2e;                // softmax scale * log2(e)
  float* ws_ml;              // partials: [items][64 rows][2]
  float* ws_o;               // partials: [items][64 rows][D]
  int32_t* item_pre;         // [B + 1] prefix sums of work items per sequence
  int64_t max_items;
  unsigned int* status;
};

// 2^e as fp32 for e in [-149, 127], 0 below.
__device__ __forceinline__ float pow2f(int e) {
  if (e >= -126) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  if (e >= -149) return __uint_as_float(1u << (e + 149));
  return 0.f;
}

// Row tiles of sequence b: ceil(n_b * G / 64).
__device__ __forceinline__ int row_tiles(int n, int G) { return (n * G + kPRows - 1) / kPRows; }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Byte offset of 16-byte chunk `ch` of row `row` in an f16 tile of D columns:
// the chunk index is XORed with the row's low 3 bits, so the 8 rows an
// ldmatrix reads at one logical chunk fall into 8 different bank groups.
template <int D>
__device__ __forceinline__ uint32_t tile_off(int row, int ch) {
  return static_cast<uint32_t>(row * (D * 2) + ((ch ^ (row & 7)) << 4));
}

}  // namespace

namespace {

// Work items: for every sequence b, kv head, row tile and key split one item,
// in that order; item_pre[b] counts the items of sequences before b.
__global__ void prefill_plan_kernel(const int32_t* cu_q, int B, int G, int Hkv, int splits, int32_t* item_pre) {
  const int lane = threadIdx.x;
  int run = 0;
  if (lane == 0) item_pre[0] = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    int x = 0;
    if (b < B) {
      const int n = max(0, cu_q[b + 1] - cu_q[b]);
      x = Hkv * row_tiles(n, G) * splits;
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (b < B) item_pre[b + 1] = run + x;
    run += __shfl_sync(kFull, x, 31);
  }
}

template <int D>
__global__ void __launch_bounds__(kPThreads, 3) prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = PC<D>;
  constexpr int NG = C::NG;
  constexpr int NKS = D / 16;  // QK k-steps
  constexpr int NNB = D / 8;   // P.V n-blocks (8 channels each)
  constexpr int HNB = NNB / 2; // n-blocks per P.V half
  constexpr int KW = C::KROW / 4;  // code words per row
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* raw = sm;
  float* ksc = reinterpret_cast<float*>(sm + C::OFF_S);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_B);
  int* s_rvt = reinterpret_cast<int*>(sm + C::OFF_B + 8 * kPNST);  // [2] tile max V byte
  int* s_badpos = s_rvt + 2;                                     // first key with a 0xFF byte
  const uint32_t kf_u32 = smem_u32(sm + C::OFF_K), vf_u32 = smem_u32(sm + C::OFF_V);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane >> 2, c = lane & 3;
  if (tid == 0) {
    for (int s = 0; s < kPNST; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    s_rvt[0] = s_rvt[1] = 0;
  }
  __syncthreads();
  pdl_wait();
  int64_t total = p.item_pre[p.B];
  if (total > p.max_items) {  // cu_q inconsistent with num_q_tokens: do nothing
    if (blockIdx.x == 0 && tid == 0) record_error(p.status, kErrBounds);
    total = 0;
  }
  const int cap = p.max_pages << p.ps_log2;
  uint32_t git = 0;  // tiles through the ring so far (stage and parity)

  for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
    // ---- which sequence, kv head, row tile and key split
    int lb = 1, hb = p.B;  // first b + 1 with item_pre[b + 1] > item
    while (lb < hb) {
      const int mid = (lb + hb) >> 1;
      if (p.item_pre[mid] > item) hb = mid; else lb = mid + 1;
    }
    const int b = lb - 1;
    const int q0 = p.cu_q[b], n_plan = max(0, p.cu_q[b + 1] - q0);  // the plan's row count
    int L = p.seq_lens[b];
    int n = n_plan;
    if (L < 0 || L > cap || n > L || q0 < 0 || q0 + n > p.T) {
      if (tid == 0) record_error(p.status, kErrBounds);
      L = L < 0 ? 0 : (L > cap ? cap : L);
      n = n > L ? L : n;
      if (q0 < 0 || q0 + n > p.T) n = 0;
    }
    const int ctx = L - n;  // keys before the chunk
    const int tiles_b = row_tiles(n_plan, p.G);
    const int64_t local = item - p.item_pre[b];
    const int kvh = static_cast<int>(local / (static_cast<int64_t>(tiles_b) * p.splits));
    const int rem = static_cast<int>(local - static_cast<int64_t>(kvh) * tiles_b * p.splits);
    const int rtile = rem / p.splits, split = rem - rtile * p.splits;
    const int row0 = rtile * kPRows;
    const int nrows = n * p.G;
    const int last_row = min(row0 + kPRows, nrows) - 1;
    const int pos_max = ctx + last_row / p.G;  // the tile's last query position
    const int k_lo = split * p.kchunk;
    const int k_hi = min(k_lo + p.kchunk, pos_max + 1);
    // this warp's rows r and r + 8
    const int wr0 = row0 + warp * 16 + r, wr1 = wr0 + 8;
    const int pos0 = wr0 < nrows ? ctx + wr0 / p.G : -1;
    const int pos1 = wr1 < nrows ? ctx + wr1 / p.G : -1;
    float* ml_out = p.ws_ml + item * (kPRows * 2);
    float* o_out = p.ws_o + item * (static_cast<int64_t>(kPRows) * D);
    if (k_lo >= k_hi) {  // the split lies past every row's position: an empty partial
      if (tid < kPRows) {
        ml_out[2 * tid] = -INFINITY;
        ml_out[2 * tid + 1] = 0.f;
      }
      continue;
    }
    const int ntiles = (k_hi - k_lo + kKT - 1) / kKT;
    const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.max_pages;
    const int lp_last = (L - 1) >> p.ps_log2;  // last page of the sequence

    // ---- producer: lanes of warp 0 issue one tile's bulk copies, one copy each
    auto issue = [&](int t) {
      const int st = (git + t) % kPNST;
      uint8_t* base = raw + st * C::RAW;
      constexpr int R0 = 16;
      const int rows_per = min(1 << p.ps_log2, kKT);  // rows of one page run
      const int runs = kKT / rows_per;
      if (lane == 0) mbar_arrive_expect_tx(&bars[st], C::RAW);
      __syncwarp();
      if (lane < 4 * runs) {
        const int run = lane >> 2, what = lane & 3;  // 0 K codes, 1 V codes, 2 K scales, 3 V scales
        const int key = k_lo + t * kKT + run * rows_per;
        int lp = key >> p.ps_log2;
        lp = lp > lp_last ? lp_last : lp;  // keys past the sequence: any page of it (masked)
        int page = bt_row[lp];
        if (page < 0 || page >= p.num_pages) {
          record_error(p.status, kErrBounds);
          page = 0;
        }
        const int64_t row = ((static_cast<int64_t>(page) * p.Hkv + kvh) << p.ps_log2) + (key & ((1 << p.ps_log2) - 1));
        const int rb = what < 2 ? C::KROW : C::SROW;
        const uint8_t* src = (what == 0 ? p.kc : what == 1 ? p.vc : what == 2 ? p.ks : p.vs) + row * rb;
        const int dst = (what < 2 ? what * kKT * C::KROW : 2 * kKT * C::KROW + (what - 2) * kKT * C::SROW) +
                        run * rows_per * rb;
        bulk_g2s(base + dst, src, static_cast<uint32_t>(rows_per * rb), &bars[st]);
      }
      (void)R0;
    };
    if (warp == 0) {
      fence_proxy_async();
      for (int t = 0; t < (ntiles < kPNST ? ntiles : kPNST); ++t) issue(t);
    }
    if (tid == 0) *s_badpos = 0x7FFFFFFF;

    // ---- the warp's 16 query rows: rotated E4M3 bytes -> f16 A fragments
    uint32_t qa[NKS][4];
    {
      uint8_t* qs = sm + C::OFF_Q + warp * C::QB;
      constexpr int CH = D / 16;  // 16-byte chunks per row
      for (int idx = lane; idx < 16 * CH; idx += 32) {
        const int rr = idx / CH, ch = idx - rr * CH, row = row0 + warp * 16 + rr;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < nrows) {
          const int64_t qrow = (static_cast<int64_t>(q0) + row / p.G) * p.Hq + kvh * p.G + row % p.G;
          v = *reinterpret_cast<const uint4*>(p.qbytes + qrow * D + ch * 16);
        }
        *reinterpret_cast<uint4*>(qs + rr * D + ch * 16) = v;
      }
      __syncwarp();
#pragma unroll
      for (int ks = 0; ks < NKS; ++ks) {
        qa[ks][0] = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(qs + r * D + 16 * ks + 2 * c));
        qa[ks][1] = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(qs + (r + 8) * D + 16 * ks + 2 * c));
        qa[ks][2] = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(qs + r * D + 16 * ks + 2 * c + 8));
        qa[ks][3] = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(qs + (r + 8) * D + 16 * ks + 2 * c + 8));
      }
    }
    __syncthreads();  // s_badpos set; every warp past its previous item's last tile

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float O[NNB][4];
#pragma unroll
    for (int nb = 0; nb < NNB; ++nb) O[nb][0] = O[nb][1] = O[nb][2] = O[nb][3] = 0.f;
    int RV = 0;  // running maximum V scale byte of this item (the same in every thread)
    bool aborted = false;

    for (int t = 0; t < ntiles; ++t) {
      const int st = (git + t) % kPNST;
      const uint8_t* rk = raw + st * C::RAW;
      const uint8_t* rv = rk + kKT * C::KROW;
      const uint8_t* rks = rv + kKT * C::KROW;
      const uint8_t* rvs = rks + kKT * C::SROW;
      const int kbase = k_lo + t * kKT;
      const bool ok = mbar_wait(&bars[st], ((git + t) / kPNST) & 1, kWaitBudget);
      if (!__syncthreads_and(ok)) {  // a copy never landed: record, drain and give up on the launch
        if (tid == 0) {
          record_error(p.status, kErrTimeout);
          for (int k = t; k < (ntiles < t + kPNST ? ntiles : t + kPNST); ++k)
            mbar_wait(&bars[(git + k) % kPNST], ((git + k) / kPNST) & 1, kWaitBudget);
        }
        aborted = true;
        break;
      }
      // phase A: the tile's largest V scale byte and its first non-finite group, over valid keys
      const int slot = t & 1;
      if (tid < kKT) {
        const int key = kbase + tid;
        if (key < k_hi) {
          int vmax = 0, bad = 0;
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const int kb = rks[tid * C::SROW + g], vb = rvs[tid * C::SROW + g];
            vmax = max(vmax, vb);
            bad |= (kb == 0xFF) | (vb == 0xFF);
          }
          atomicMax(&s_rvt[slot], vmax);
          if (bad) atomicMin(s_badpos, key);
        }
      }
      __syncthreads();
      const int RVn = max(RV, s_rvt[slot]);
      const float rvf = pow2f(RV - RVn);  // rescale of O when the reference grows
      RV = RVn;
      if (tid == 0) s_rvt[slot ^ 1] = 0;
      // phase B: the tile in f16 -- K codes (exact) in natural channel order,
      // V codes times 2^(byte - RV); keys past the range are zero in V
      for (int wi = tid; wi < kKT * KW; wi += kPThreads) {
        const int tok = wi / KW, pos = wi - tok * KW;
        uint32_t h[4];
        e2m1x8_to_f16x2(reinterpret_cast<const uint32_t*>(rk)[wi], h);
        const int g = pos % NG, w = pos / NG;  // K rows: word w of group g at position NG*w + g
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(kf_u32 + tile_off<D>(tok, 4 * g + w)),
                     "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]) : "memory");
        uint32_t v[4] = {0u, 0u, 0u, 0u};
        if (kbase + tok < k_hi) {
          const int vbyte = rvs[tok * C::SROW + pos / 4];
          const float f = pow2f(vbyte - RV);
          const uint32_t f2 = pack_f16x2(f, f);
          e2m1x8_to_f16x2(reinterpret_cast<const uint32_t*>(rv)[wi], v);
#pragma unroll
          for (int k = 0; k < 4; ++k) v[k] = hmul2(v[k], f2);
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(vf_u32 + tile_off<D>(tok, pos)),
                     "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]) : "memory");
      }
      for (int i = tid; i < NG * kKT; i += kPThreads) {
        const int g = i / kKT, tok = i - g * kKT;
        ksc[i] = __uint_as_float(static_cast<uint32_t>(rks[tok * C::SROW + g]) << 23);  // 2^(byte-127); 0 -> 0
      }
      __syncthreads();
      if (warp == 0 && t + kPNST < ntiles) {  // the raw stage is free again
        fence_proxy_async();
        issue(t + kPNST);
      }
      // phase C: this warp's 16 rows against the tile's 64 keys, in two
      // sub-tiles of 32 keys (fewer live registers: S, P and the QK
      // accumulators cover 32 keys at a time)
#pragma unroll 1
      for (int sub = 0; sub < 2; ++sub) {
        const int kb0 = kbase + 32 * sub;
        float S[4][4];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          float acc[4][4];
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const int ks = 2 * g + kk;
#pragma unroll
            for (int nbp = 0; nbp < 2; ++nbp) {
              const int mi = lane >> 3, tok = 32 * sub + 8 * (2 * nbp + (mi >> 1)) + (lane & 7);
              uint32_t b0, b1, b2, b3;
              ldsm_x4(kf_u32 + tile_off<D>(tok, 2 * ks + (mi & 1)), b0, b1, b2, b3);
              if (kk == 0) {
                mma_f16_zc(acc[2 * nbp], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                mma_f16_zc(acc[2 * nbp + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
              } else {
                mma_f16(acc[2 * nbp], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                mma_f16(acc[2 * nbp + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
              }
            }
          }
#pragma unroll
          for (int nb = 0; nb < 4; ++nb) {
            const float2 f = *reinterpret_cast<const float2*>(ksc + g * kKT + 32 * sub + 8 * nb + 2 * c);
            if (g == 0) {
              S[nb][0] = acc[nb][0] * f.x; S[nb][1] = acc[nb][1] * f.y;
              S[nb][2] = acc[nb][2] * f.x; S[nb][3] = acc[nb][3] * f.y;
            } else {
              S[nb][0] = fmaf(acc[nb][0], f.x, S[nb][0]); S[nb][1] = fmaf(acc[nb][1], f.y, S[nb][1]);
              S[nb][2] = fmaf(acc[nb][2], f.x, S[nb][2]); S[nb][3] = fmaf(acc[nb][3], f.y, S[nb][3]);
            }
          }
        }
        // causal and range mask, online softmax (exact running max per row)
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
          const int key = kb0 + 8 * nb + 2 * c;
          S[nb][0] = (key <= pos0 && key < k_hi) ? S[nb][0] * p.sl2e : -INFINITY;
          S[nb][1] = (key + 1 <= pos0 && key + 1 < k_hi) ? S[nb][1] * p.sl2e : -INFINITY;
          S[nb][2] = (key <= pos1 && key < k_hi) ? S[nb][2] * p.sl2e : -INFINITY;
          S[nb][3] = (key + 1 <= pos1 && key + 1 < k_hi) ? S[nb][3] * p.sl2e : -INFINITY;
          mx0 = fmaxf(mx0, fmaxf(S[nb][0], S[nb][1]));
          mx1 = fmaxf(mx1, fmaxf(S[nb][2], S[nb][3]));
        }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
        }
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float a0 = n0 == -INFINITY ? 1.f : ex2(m0 - n0), a1 = n1 == -INFINITY ? 1.f : ex2(m1 - n1);
        const float base0 = n0 == -INFINITY ? 0.f : n0, base1 = n1 == -INFINITY ? 0.f : n1;
        m0 = n0;
        m1 = n1;
        const float o0 = sub == 0 ? a0 * rvf : a0, o1 = sub == 0 ? a1 * rvf : a1;
#pragma unroll
        for (int nb = 0; nb < NNB; ++nb) {
          O[nb][0] *= o0; O[nb][1] *= o0; O[nb][2] *= o1; O[nb][3] *= o1;
        }
        float s0 = 0.f, s1 = 0.f;
        uint32_t ph[2][4], pl[2][4];  // P as A fragments of the sub-tile's 2 key k-steps, hi and lo parts
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
          const float q0 = ex2(S[nb][0] - base0), q1 = ex2(S[nb][1] - base0);
          const float q2 = ex2(S[nb][2] - base1), q3 = ex2(S[nb][3] - base1);
          s0 += q0 + q1;
          s1 += q2 + q3;
          const float h0 = __uint_as_float(__float_as_uint(q0) & 0xFFFFE000u);
          const float h1 = __uint_as_float(__float_as_uint(q1) & 0xFFFFE000u);
          const float h2 = __uint_as_float(__float_as_uint(q2) & 0xFFFFE000u);
          const float h3 = __uint_as_float(__float_as_uint(q3) & 0xFFFFE000u);
          const int j = nb >> 1, hi = (nb & 1) * 2;  // n-block 2j -> a0, a1; 2j+1 -> a2, a3
          ph[j][hi] = pack_f16x2(h0, h1);
          ph[j][hi + 1] = pack_f16x2(h2, h3);
          pl[j][hi] = pack_f16x2(q0 - h0, q1 - h1);
          pl[j][hi + 1] = pack_f16x2(q2 - h2, q3 - h3);
        }
        l0 = l0 * a0 + s0;
        l1 = l1 * a1 + s1;
        // P.V in two halves of the channels, each sub-tile into a fresh accumulator
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float acc[HNB][4];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int nbp = 0; nbp < HNB / 2; ++nbp) {
              const int nbA = half * HNB + 2 * nbp;
              const int mi = lane >> 3, tok = 32 * sub + 16 * j + 8 * (mi & 1) + (lane & 7);
              uint32_t b0, b1, b2, b3;
              ldsm_x4_t(vf_u32 + tile_off<D>(tok, nbA + (mi >> 1)), b0, b1, b2, b3);
              if (j == 0) {
                mma_f16_zc(acc[2 * nbp], ph[j][0], ph[j][1], ph[j][2], ph[j][3], b0, b1);
                mma_f16_zc(acc[2 * nbp + 1], ph[j][0], ph[j][1], ph[j][2], ph[j][3], b2, b3);
              } else {
                mma_f16(acc[2 * nbp], ph[j][0], ph[j][1], ph[j][2], ph[j][3], b0, b1);
                mma_f16(acc[2 * nbp + 1], ph[j][0], ph[j][1], ph[j][2], ph[j][3], b2, b3);
              }
              mma_f16(acc[2 * nbp], pl[j][0], pl[j][1], pl[j][2], pl[j][3], b0, b1);
              mma_f16(acc[2 * nbp + 1], pl[j][0], pl[j][1], pl[j][2], pl[j][3], b2, b3);
            }
          }
#pragma unroll
          for (int i = 0; i < HNB; ++i) {
            add2(O[half * HNB + i][0], O[half * HNB + i][1], acc[i][0], acc[i][1]);
            add2(O[half * HNB + i][2], O[half * HNB + i][3], acc[i][2], acc[i][3]);
          }
        }
      }
      __syncthreads();  // the f16 tiles may be overwritten
    }
    if (aborted) break;
    git += ntiles;
    // ---- partial of this (row tile, key split): m, l (quad-reduced) and unnormalised O
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, o);
      l1 += __shfl_xor_sync(kFull, l1, o);
    }
    const int badpos = *s_badpos;  // rows that see a non-finite group are NaN
    if (pos0 >= badpos) l0 = __int_as_float(0x7FC00000);
    if (pos1 >= badpos) l1 = __int_as_float(0x7FC00000);
    const float osc = pow2f(RV - 127);  // V was taken as code * 2^(byte - RV)
    const int lr0 = warp * 16 + r, lr1 = lr0 + 8;
    if (c == 0) {
      ml_out[2 * lr0] = m0;
      ml_out[2 * lr0 + 1] = l0;
      ml_out[2 * lr1] = m1;
      ml_out[2 * lr1 + 1] = l1;
    }
#pragma unroll
    for (int nb = 0; nb < NNB; ++nb) {
      *reinterpret_cast<float2*>(o_out + lr0 * D + 8 * nb + 2 * c) = make_float2(O[nb][0] * osc, O[nb][1] * osc);
      *reinterpret_cast<float2*>(o_out + lr1 * D + 8 * nb + 2 * c) = make_float2(O[nb][2] * osc, O[nb][3] * osc);
    }
  }
  pdl_trigger();
}

struct PrefillMergeParams {
  const float* ws_ml;
  const float* ws_o;
  const int32_t* item_pre;
  const int32_t* cu_q;
  const int32_t* seq_lens;
  int B, T, Hq, G, splits, cap;
  int64_t max_items;
  float* out;
  uqh::SignMasks sign;
};

// One warp per (query token, query head): log-sum-exp merge of the row's key
// splits, normalisation, then the inverse rotation s .* (H o) / sqrt(D) with
// the butterfly strides below D/32 inside a lane and the rest across lanes.
template <int D>
__global__ void __launch_bounds__(128) prefill_merge_kernel(const __grid_constant__ PrefillMergeParams p) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (row >= static_cast<int64_t>(p.T) * p.Hq) return;
  const int t = static_cast<int>(row / p.Hq), h = static_cast<int>(row - static_cast<int64_t>(t) * p.Hq);
  int lb = 1, hb = p.B;  // sequence b: cu_q[b] <= t < cu_q[b + 1]
  while (lb < hb) {
    const int mid = (lb + hb) >> 1;
    if (p.cu_q[mid] > t) hb = mid; else lb = mid + 1;
  }
  const int b = lb - 1;
  const int q0 = p.cu_q[b], n_plan = max(0, p.cu_q[b + 1] - q0);
  int L = p.seq_lens[b], n = n_plan;
  L = L < 0 ? 0 : (L > p.cap ? p.cap : L);
  n = n > L ? L : n;
  if (q0 < 0 || q0 + n > p.T || p.item_pre[p.B] > p.max_items) n = 0;
  const int i = t - q0;
  float o[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) o[e] = 0.f;
  if (i >= 0 && i < n) {
    const int kvh = h / p.G, hl = h - kvh * p.G;
    const int rowi = i * p.G + hl, rtile = rowi / kPRows, rr = rowi - rtile * kPRows;
    const int64_t item0 = p.item_pre[b] + (static_cast<int64_t>(kvh) * row_tiles(n_plan, p.G) + rtile) * p.splits;
    float Ms = -INFINITY;
    for (int s0 = 0; s0 < p.splits; s0 += 32) {
      const int s = s0 + lane;
      if (s < p.splits) Ms = fmaxf(Ms, p.ws_ml[((item0 + s) * kPRows + rr) * 2]);
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) Ms = fmaxf(Ms, __shfl_xor_sync(kFull, Ms, k));
    float Ls = 0.f;
    for (int s0 = 0; s0 < p.splits; s0 += 32) {
      const int s = s0 + lane;
      float w = 0.f;
      bool live = false;
      if (s < p.splits) {
        const float m = p.ws_ml[((item0 + s) * kPRows + rr) * 2];
        live = m != -INFINITY;  // an empty split wrote no output row
        if (live) {
          w = ex2(m - Ms);
          Ls += w * p.ws_ml[((item0 + s) * kPRows + rr) * 2 + 1];
        }
      }
      const unsigned mask = __ballot_sync(kFull, live);
      const int cnt = min(32, p.splits - s0);
      for (int j = 0; j < cnt; ++j) {
        const float wj = __shfl_sync(kFull, w, j);
        if ((mask >> j) & 1u) {
          const float* src = p.ws_o + ((item0 + s0 + j) * kPRows + rr) * D + lane * EPL;
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[e] += wj * src[e];
        }
      }
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) Ls += __shfl_xor_sync(kFull, Ls, k);
    const float inv = 1.f / Ls;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] *= inv;
#pragma unroll
    for (int hs = 1; hs < EPL; hs <<= 1)
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        if ((e & hs) == 0) {
          const float x = o[e], y = o[e + hs];
          o[e] = x + y;
          o[e + hs] = x - y;
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
    for (int e = 0; e < EPL; ++e) o[e] = __uint_as_float(__float_as_uint(o[e] * sc) ^ p.sign.m[lane * EPL + e]);
  }
  float* dst = p.out + row * D + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; ++e) dst[e] = o[e];
}

}  // namespace

// ------------------------------------------------------------------ host
namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct PrefillPlan {
  int splits, kchunk;
  int64_t max_items;
  size_t off_pre, off_q, off_ml, off_o, total;
};

PrefillPlan plan_prefill(int T, int B, int hq, int hkv, int d, int max_keys, int sms) {
  PrefillPlan pl;
  const int G = hq / hkv;
  const int64_t tiles = (static_cast<int64_t>(T) * G + kPRows - 1) / kPRows + B;  // bound on row tiles per kv head
  const int64_t base = static_cast<int64_t>(hkv) * tiles;
  const int64_t target = 2LL * 2 * sms;  // two waves of two blocks per SM
  const int max_splits = std::max(1, (max_keys + kKT - 1) / kKT);
  pl.splits = static_cast<int>(std::min<int64_t>(max_splits, std::max<int64_t>(1, (target + base - 1) / base)));
  pl.kchunk = ((max_keys + pl.splits - 1) / pl.splits + kKT - 1) / kKT * kKT;
  pl.max_items = base * pl.splits;
  pl.off_pre = 256;
  pl.off_q = pl.off_pre + align256(static_cast<size_t>(B + 1) * 4);
  pl.off_ml = pl.off_q + align256(static_cast<size_t>(T) * hq * d);
  pl.off_o = pl.off_ml + align256(static_cast<size_t>(pl.max_items) * kPRows * 2 * 4);
  pl.total = pl.off_o + static_cast<size_t>(pl.max_items) * kPRows * d * 4;
  return pl;
}

template <int D>
uq_status run_prefill(const uqh::PrefillArgs& a, cudaStream_t s) {
  using C = PC<D>;
  const uq_cache& c = *a.cache;
  const uqh::DevInfo& di = uqh::dev_info();
  const int G = a.num_q_heads / c.num_kv_heads;
  const PrefillPlan pl = plan_prefill(a.num_q_tokens, a.batch, a.num_q_heads, c.num_kv_heads, D,
                                      a.max_pages * c.page_size, di.sms);
  if (a.ws_bytes < pl.total) return UQ_ERR_WORKSPACE;
  auto kern = prefill_kernel<D>;
  static int cfg_dev = -1;
  static int per_sm = 0;
  if (cfg_dev != di.device) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return UQ_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPThreads, C::SMEM) != cudaSuccess || per_sm < 1)
      return UQ_ERR_CUDA;
    cfg_dev = di.device;
  }
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  PrefillParams p;
  p.qbytes = ws + pl.off_q;
  p.cu_q = a.cu_q;
  p.seq_lens = a.seq_lens;
  p.block_table = a.block_table;
  p.max_pages = a.max_pages;
  p.kc = static_cast<const uint8_t*>(c.k_codes);
  p.ks = static_cast<const uint8_t*>(c.k_scales);
  p.vc = static_cast<const uint8_t*>(c.v_codes);
  p.vs = static_cast<const uint8_t*>(c.v_scales);
  p.B = a.batch;
  p.T = a.num_q_tokens;
  p.Hq = a.num_q_heads;
  p.Hkv = c.num_kv_heads;
  p.G = G;
  p.ps_log2 = uqh::ilog2(c.page_size);
  p.num_pages = c.num_pages;
  p.splits = pl.splits;
  p.kchunk = pl.kchunk;
  const float sm = a.sm_scale > 0.f ? a.sm_scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  p.sl2e = sm * 1.4426950408889634f;
  p.ws_ml = reinterpret_cast<float*>(ws + pl.off_ml);
  p.ws_o = reinterpret_cast<float*>(ws + pl.off_o);
  p.item_pre = reinterpret_cast<int32_t*>(ws + pl.off_pre);
  p.max_items = pl.max_items;
  p.status = uqh::status_word();
  if (!p.status) return UQ_ERR_CUDA;

  prefill_plan_kernel<<<1, 32, 0, s>>>(a.cu_q, a.batch, G, c.num_kv_heads, pl.splits, p.item_pre);
  if (cudaGetLastError() != cudaSuccess) return UQ_ERR_CUDA;
  const uq_status st = uqh::launch_test_query_fp8(a.q, static_cast<int64_t>(a.num_q_tokens) * a.num_q_heads, D,
                                                  c.rot_seed, ws + pl.off_q, s);
  if (st != UQ_OK) return st;
  const int64_t grid = std::min<int64_t>(pl.max_items, static_cast<int64_t>(di.sms) * per_sm);
  if (uqh::launch_pdl(kern, static_cast<unsigned>(std::max<int64_t>(grid, 1)), kPThreads, C::SMEM, s, p) !=
      cudaSuccess)
    return UQ_ERR_CUDA;
  PrefillMergeParams mp;
  mp.ws_ml = p.ws_ml;
  mp.ws_o = p.ws_o;
  mp.item_pre = p.item_pre;
  mp.cu_q = a.cu_q;
  mp.seq_lens = a.seq_lens;
  mp.B = a.batch;
  mp.T = a.num_q_tokens;
  mp.Hq = a.num_q_heads;
  mp.G = G;
  mp.splits = pl.splits;
  mp.max_items = pl.max_items;
  mp.cap = a.max_pages * c.page_size;
  mp.out = a.out;
  uqh::make_sign_masks(c.rot_seed, D, &mp.sign);
  const int64_t rows = static_cast<int64_t>(a.num_q_tokens) * a.num_q_heads;
  return uqh::cuda_status(
      uqh::launch_pdl(prefill_merge_kernel<D>, static_cast<unsigned>((rows + 3) / 4), 128, 0, s, mp));
}

}  // namespace

namespace uqh {

size_t prefill_workspace_bytes(int T, int B, int hq, int hkv, int d, int max_keys) {
  return plan_prefill(T, B, hq, hkv, d, max_keys, std::max(1, dev_info().sms)).total;
}

uq_status launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  return a.cache->head_dim == 128 ? run_prefill<128>(a, s) : run_prefill<64>(a, s);
}

}  // namespace uqh
