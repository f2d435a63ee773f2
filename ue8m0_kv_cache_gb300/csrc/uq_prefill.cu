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
//   * A work item is 128 query rows of one (sequence, kv head) -- consecutive
//     (token, head) pairs of the chunk, one row per tensor-memory lane -- and
//     one range of keys, in tiles of 64 keys.  The page rows of a tile's K
//     codes, V codes and both scale rows are copied by 16-byte cp.async into a
//     ring of raw stages.
//   * QK^T runs on the block-scaled tensor-core path the pages' kernel uses
//     (§4.2: the matrix unit consumes the FP4 codes and their UE8M0 scale
//     bytes directly): tcgen05.mma kind::mxf8f6f4 with A = the E4M3 query rows,
//     B = the tile's E2M1 K codes, one MMA per 32-channel group, the keys'
//     scale bytes as the B scale factors in tensor memory (the query's are 1).
//     The K codes are only repacked (the cache interleaves their words by
//     group; the operand wants natural order, 16 codes per 16-byte chunk);
//     no K value is ever widened.
//   * V' = code * 2^(byte - RV) MN-major (channels contiguous, RV the item's
//     running maximum V byte), converted once per tile for all 128 rows: the
//     V scale varies along the P.V contraction (keys), so it cannot be a
//     block scale of that MMA.  Exact in f16 except where a V group lies so
//     far below RV that its values underflow.
//   * Each row's logits are read from tensor memory, masked (causal), and go
//     through the online softmax (lazy running maximum); P goes back over S
//     as hi and lo f16 parts, and O_win += P V' runs with A from tensor
//     memory.  O_win sums a window of up to sixteen tiles under one reference
//     (running max, RV) and is then added to the row's fp32 O with IEEE
//     rounding, as the decode adds its per-unit partials.
//   * Two kernels do this.  prefill_ws_kernel (head_dim 128, the default)
//     gives each stage warps of its own -- copy, V statistics and operand
//     conversion, softmax, and one thread each issuing QK^T and P.V -- with O
//     in tensor memory and S/P and the operands double-buffered, one CTA per
//     SM.  prefill_tc_kernel (head_dim 64, or UQ_PREFILL=tc) runs every stage
//     in the same 4 warps, O in registers, two CTAs per SM.
//   * Long key ranges are split over work items; each (row tile, key split)
//     writes a partial (m, l, O) and a merge kernel combines them by
//     log-sum-exp and applies the inverse rotation.
#include <algorithm>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <cmath>
#include <mutex>

#include "uq_device.cuh"
#include "uq_internal.h"
#include "uq_tc.cuh"

namespace {

using namespace uqd;
using namespace uqtc;

constexpr int kPThreads = 128;  // 4 warps: one query row per thread
constexpr int kTileKeys = 64;   // keys per tile; key splits are whole tiles
constexpr int kMergeOneRound = 8;  // the merge loads up to this many splits' partials in one round
constexpr int kItemCost = 3;    // per-item cost in key tiles, for the split choice (fitted to measured times)

struct PrefillParams {
  const uint8_t* qbytes;     // rotated E4M3 query, [T][Hq][D]
  const int32_t* cu_q;       // [B + 1] first query token of each sequence (cascade: of each group)
  const int32_t* seq_lens;   // [B] keys of each sequence after the chunk (cascade: shared prefix of each group)
  const int32_t* block_table;
  int max_pages;
  const uint8_t* kc;
  const uint8_t* ks;
  const uint8_t* vc;
  const uint8_t* vs;
  int B, T, Hq, Hkv, G, ps_log2, num_pages;
  float sl2e;                // softmax scale * log2(e)
  float* ws_ml;              // partials: [items][128 rows][2]
  float* ws_o;               // partials: [items][128 rows][D]
  int32_t* item_pre;         // [B + 1] prefix sums of work items per sequence, then S and keys per split
  int64_t max_items;
  unsigned int* status;
  // Cascade mode: "sequence" b is group b, its queries are the decode queries of
  // sequences cu_q[b] .. cu_q[b+1]-1 (T = batch), its keys the group's shared
  // prefix from the block-table row of its first sequence, attended without a
  // causal mask.
  int cascade, min_rows, casc_cap;
};

// 2^e as fp32 for e in [-149, 127], 0 below.
__device__ __forceinline__ float pow2f(int e) {
  if (e >= -126) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  if (e >= -149) return __uint_as_float(1u << (e + 149));
  return 0.f;
}

// Row tiles of sequence b: ceil(n_b * G / rows), rows the query rows of one work item.
__device__ __forceinline__ int row_tiles(int n, int G, int rows) { return (n * G + rows - 1) / rows; }

}  // namespace

namespace {

// Work items: for every sequence b, kv head, row tile and key split one item,
// in that order; item_pre[b] counts the items of sequences before b, and
// item_pre[B + 1], item_pre[B + 2] receive the split count S and the keys per
// split.  Both come from the key ranges actually present (the longest one,
// Lmax), not from the block table's capacity: kchunk = ceil(Lmax / 64 / S) key
// tiles.  With fixed_splits > 0 (cascade: the decode's merge reads the same S)
// S is that; otherwise S in [1, max_splits] minimises the estimated time of
// the busiest CTA under the grid-stride order of the items,
// ceil(items(S) / ctas) * (tiles per split + kItemCost), kItemCost the
// per-item cost in key tiles (query staging, pipeline fill, and the 66 KB
// partial that this kernel writes and the merge reads back).
// Cascade mode (prefix != nullptr): a group whose shared keys are 0 has no items.
__global__ void prefill_plan_kernel(const int32_t* cu_q, const int32_t* keys, int B, int G, int Hkv, int max_splits,
                                    int fixed_splits, int rows, const int32_t* prefix, int min_rows, int cap,
                                    int ctas, int32_t* item_pre) {
  const int lane = threadIdx.x;
  // pass 1: row-tile units and the longest key range
  long long units = 0;
  int lmax = 0;
  for (int b = lane; b < B; b += 32) {
    const int n = max(0, cu_q[b + 1] - cu_q[b]);
    int L;
    if (prefix != nullptr) {
      L = casc_shared_keys(n, G, prefix[b], min_rows, cap);
    } else {
      L = keys[b];
      L = L < 0 ? 0 : (L > cap ? cap : L);
    }
    if (prefix == nullptr || L > 0) units += static_cast<long long>(Hkv) * row_tiles(n, G, rows);
    lmax = max(lmax, L);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    units += __shfl_xor_sync(kFull, units, o);
    lmax = max(lmax, __shfl_xor_sync(kFull, lmax, o));
  }
  const int kt = max(1, (lmax + kTileKeys - 1) / kTileKeys);
  int splits = fixed_splits;
  if (splits < 1) {
    const int smax = max(1, min(min(max_splits, kt), 0xFFFFF));
    long long best = LLONG_MAX;  // (cost << 20) | S: ties go to the smaller S
    for (int s0 = 1; s0 <= smax; s0 += 32) {
      const int S = s0 + lane;
      if (S <= smax) {
        const long long waves = (units * S + ctas - 1) / ctas;
        const long long key = ((waves * ((kt + S - 1) / S + kItemCost)) << 20) | S;
        best = min(best, key);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = min(best, __shfl_xor_sync(kFull, best, o));
    splits = static_cast<int>(best & 0xFFFFF);
  }
  const int kchunk = (kt + splits - 1) / splits * kTileKeys;
  // pass 2: prefix sums of the items
  int run = 0;
  if (lane == 0) {
    item_pre[0] = 0;
    item_pre[B + 1] = splits;
    item_pre[B + 2] = kchunk;
  }
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    int x = 0;
    if (b < B) {
      const int n = max(0, cu_q[b + 1] - cu_q[b]);
      const bool live = prefix == nullptr || casc_shared_keys(n, G, prefix[b], min_rows, cap) > 0;
      x = live ? Hkv * row_tiles(n, G, rows) * splits : 0;
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

// ------------------------------------------------------------ tensor-memory (tcgen05) kernel
constexpr int kTRows = 128;     // query rows per CTA
constexpr int kTKT = kTileKeys; // keys per tile
constexpr int kTNST = 3;        // raw stages
constexpr int kTWin = 16;       // tiles per O window
// Tensor memory columns: S [0,64) (the tile's P hi [0,32) and P lo [32,64) overwrite
// it once read), the query scale factors [64,68), the key scale factors [96,98),
// O_win [128, 128 + D).  Scale-factor columns start on 32-column boundaries.
constexpr int kTCols = 256;
constexpr int kSfaCol = 64;
constexpr int kSfbCol = 96;
// The running max is raised only when a logit exceeds it by more than this
// (log2 units).  P = 2^(x - max) then stays below 2^14, inside f16 with the hi
// part exact.  A raise closes the P.V window for the whole 128-row tile, and
// the logits' spread (a std of ~7 log2 units with rotated outlier channels)
// made a slack of 8 close it on most tiles.
constexpr float kTSlack = 14.f;

template <int D>
struct TC {
  static constexpr int KROW = D / 2, SROW = D / 32, NG = D / 32;
  static constexpr int RAW = 2 * kTKT * KROW + 2 * kTKT * SROW;
  static constexpr int QB = kTRows * 128;           // Q, E4M3, [row][128 B] (D = 64 uses half of each row)
  static constexpr int KB = kTKT * 128;              // K, E2M1 padded (16 codes in 8 of every 16 bytes), [key][128 B]
  static constexpr int VB = kTKT * 2 * D;            // V', f16, MN-major: [atom][key][128 B = 64 channels]
  static constexpr int OFF_Q = 0;                    // operands first: 1024-byte aligned
  static constexpr int OFF_K = OFF_Q + QB;
  static constexpr int OFF_V = OFF_K + KB;
  static constexpr int OFF_RAW = OFF_V + VB;
  static constexpr int OFF_BAR = OFF_RAW + kTNST * RAW;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;    // barriers and block state, + slack for the 1024-byte alignment
};

// kind::f16 instruction descriptors: D f32, A and B f16, A K-major, B K-major
// or (b_mn) MN-major, M 128.
constexpr uint32_t tc_idesc(int n, bool b_mn = false) {
  return (1u << 4) | (b_mn ? 1u << 16 : 0u) | (static_cast<uint32_t>(n >> 3) << 17) | ((128u >> 4) << 24);
}
// kind::mxf8f6f4 block-scaled descriptor: A E4M3 (format 0), B E2M1 (format 5),
// both K-major, N keys, M 128, UE8M0 scale factors (bit 23); the scale byte of
// each row and key is byte g of its 32-bit scale-factor word (A and B scale
// factor ids, bits 29-30 and 4-5), g the 32-channel group the MMA covers.
constexpr uint32_t tc_idesc_bs(int n, int g) {
  return (5u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) |
         (static_cast<uint32_t>(g) << 29) | (static_cast<uint32_t>(g) << 4);
}

// V' of a 64-key tile, MN-major in the 128-byte swizzled layout (see sw128_off):
// threads t and t ^ 1 of 128 share key row t / 2, each taking half of its
// channels, so that each thread scales whole 32-channel groups (one multiplier
// 2^(byte - RVn) per group, 0 for keys past the range and non-finite groups).
template <int D>
__device__ __forceinline__ void convert_v_half_row(const uint8_t* rv, const uint8_t* rvs, int t, bool key_ok,
                                                   int RVn, uint32_t v_dst) {
  constexpr int KROW = D / 2, SROW = D / 32, WPT = D / 16;  // code bytes per row, groups per row, words per thread
  const int key = t >> 1, hh = t & 1;
  uint32_t words[WPT];
  {
    const uint4* src = reinterpret_cast<const uint4*>(rv + key * KROW + hh * (KROW / 2));
#pragma unroll
    for (int i = 0; i < WPT / 4; ++i) {
      const uint4 w = src[i];
      words[4 * i] = w.x;
      words[4 * i + 1] = w.y;
      words[4 * i + 2] = w.z;
      words[4 * i + 3] = w.w;
    }
  }
  uint32_t mult[WPT / 4];
#pragma unroll
  for (int q2 = 0; q2 < WPT / 4; ++q2) {  // this thread's groups: hh * WPT / 4 + q2
    const int vb = rvs[key * SROW + hh * (WPT / 4) + q2];
    const float fv = (key_ok && vb != 0xFF) ? __uint_as_float(static_cast<uint32_t>(max(vb - RVn + 127, 0)) << 23)
                                            : 0.f;  // 2^(vb - RVn) <= 1; below 2^-126 far under f16's range
    mult[q2] = pack_f16x2(fv, fv);
  }
#pragma unroll
  for (int e = 0; e < WPT; ++e) {
    const int q = hh * WPT + e;  // 16-byte chunk q = channels 8q .. 8q + 7
    uint32_t hv[4];
    e2m1x8_to_f16x2(words[e], hv);
#pragma unroll
    for (int k = 0; k < 4; ++k) hv[k] = hmul2(hv[k], mult[e >> 2]);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(v_dst + sw128_off(kTKT, key, q)), "r"(hv[0]),
                 "r"(hv[1]), "r"(hv[2]), "r"(hv[3]) : "memory");
  }
}

template <int D>
__global__ void __launch_bounds__(kPThreads, 2) prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
  using C = TC<D>;
  constexpr int NG = C::NG;
  constexpr int KW = C::KROW / 4;  // code words per row
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  const uint32_t q_u32 = sb + C::OFF_Q, k_u32 = sb + C::OFF_K, v_u32 = sb + C::OFF_V;
  uint8_t* raw = sm + C::OFF_RAW;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);  // [0, kTNST) raw ring, [3] S done, [4] P.V done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 64);
  int* s_vmax = reinterpret_cast<int*>(sm + C::OFF_BAR + 72);   // [2 tiles][2 warps] tile max V byte
  int* s_bad = s_vmax + 4;                                      // [2 tiles][2 warps] first key with a 0xFF group
  float* s_sl2e = reinterpret_cast<float*>(s_bad + 4);          // the softmax scale * log2(e)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kTNST; ++s) mbar_init(&bars[s], kPThreads);  // every thread's copies arrive
    for (int s = kTNST; s < kTNST + 2; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    *s_sl2e = p.sl2e;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(kTCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = *tslot;
  const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;  // this warp's TMEM lanes
  {  // query scale factors: every query row's group scale is 1 (byte 127), in all four columns
    const uint32_t one = 0x7F7F7F7Fu;
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %1, %1, %1};" ::"r"(tmem + lanes + kSfaCol),
                 "r"(one) : "memory");
    tmem_wait_st();
  }
  pdl_wait();
  int64_t total = p.item_pre[p.B];
  const int splits = p.item_pre[p.B + 1], kchunk = p.item_pre[p.B + 2];
  if (total > p.max_items || splits < 1 || kchunk < kTKT) {
    if (blockIdx.x == 0 && tid == 0) record_error(p.status, kErrBounds);
    total = 0;
  }
  const int cap = p.max_pages << p.ps_log2;
  uint32_t git = 0, s_phase = 0, pv_phase = 0;
  bool pv_pending = false, failed = false;

  for (int64_t item = blockIdx.x; item < total && !failed; item += gridDim.x) {
    int lb = 1, hb = p.B;
    while (lb < hb) {
      const int mid = (lb + hb) >> 1;
      if (p.item_pre[mid] > item) hb = mid; else lb = mid + 1;
    }
    const int b = lb - 1;
    const int q0 = p.cu_q[b], n_plan = max(0, p.cu_q[b + 1] - q0);
    int L = p.seq_lens[b];
    int n = n_plan;
    if (p.cascade) {
      L = casc_shared_keys(n_plan, p.G, L, p.min_rows, p.casc_cap);
      if (q0 < 0 || q0 + n > p.T) {
        if (tid == 0) record_error(p.status, kErrBounds);
        L = 0;  // no keys: the item writes empty partials below
      }
    } else if (L < 0 || L > cap || n > L || q0 < 0 || q0 + n > p.T) {
      if (tid == 0) record_error(p.status, kErrBounds);
      L = L < 0 ? 0 : (L > cap ? cap : L);
      n = n > L ? L : n;
      if (q0 < 0 || q0 + n > p.T) n = 0;
    }
    const int ctx = p.cascade ? 0 : L - n;
    const int tiles_b = row_tiles(n_plan, p.G, kTRows);
    const int64_t local = item - p.item_pre[b];
    const int kvh = static_cast<int>(local / (static_cast<int64_t>(tiles_b) * splits));
    const int rem = static_cast<int>(local - static_cast<int64_t>(kvh) * tiles_b * splits);
    const int rtile = rem / splits, split = rem - rtile * splits;
    const int row0 = rtile * kTRows, nrows = n * p.G;
    const int last_row = min(row0 + kTRows, nrows) - 1;
    const int pos_max = p.cascade ? L - 1 : ctx + last_row / p.G;
    const int k_lo = split * kchunk;
    const int k_hi = min(k_lo + kchunk, pos_max + 1);
    const int my_row = row0 + tid;
    const int pos = my_row < nrows ? (p.cascade ? L - 1 : ctx + my_row / p.G) : -1;
    const int pos_lo = p.cascade ? L - 1 : ctx + row0 / p.G;  // the smallest position of the item's rows
    float* ml_out = p.ws_ml + item * (kTRows * 2);
    float* o_out = p.ws_o + item * (static_cast<int64_t>(kTRows) * D);
    if (k_lo >= k_hi) {
      ml_out[2 * tid] = -INFINITY;
      ml_out[2 * tid + 1] = 0.f;
      continue;
    }
    const int ntiles = (k_hi - k_lo + kTKT - 1) / kTKT;
    const int32_t* bt_row = p.block_table + static_cast<int64_t>(p.cascade ? q0 : b) * p.max_pages;
    const int lp_last = (L - 1) >> p.ps_log2;

    // The tile's keys come in runs of rows_per consecutive keys, one page each.
    // Lane r of every warp holds the page of run r of a tile (a global load, made
    // one tile ahead of its use); every thread then copies its share of the
    // tile with 16-byte cp.async: K and V code chunks c = tid and tid + 128
    // (rows c / 4), the scale rows' 16-byte chunks by threads 0-31, and one
    // no-increment arrival on the stage's barrier, which expects all threads.
    const int rows_per = min(1 << p.ps_log2, kTKT);
    const int rp_log2 = p.ps_log2 < 6 ? p.ps_log2 : 6;  // log2(rows_per)
    auto page_of = [&](int t) {
      int page = 0;
      if (lane < kTKT / rows_per) {
        const int key = k_lo + t * kTKT + lane * rows_per;
        int lp = key >> p.ps_log2;
        lp = lp > lp_last ? lp_last : lp;  // keys past the sequence: any page of it (masked)
        page = bt_row[lp];
      }
      return page;
    };
    auto issue = [&](int t, int page_lane) {
      const int st = (git + t) % kTNST;
      const uint32_t base = smem_u32(raw + st * C::RAW);
      const int ps_mask = (1 << p.ps_log2) - 1;
      auto row_of = [&](int r) {  // physical row of key row r of the tile
        int page = __shfl_sync(kFull, page_lane, r >> rp_log2);
        if (page < 0 || page >= p.num_pages) {
          record_error(p.status, kErrBounds);
          page = 0;
        }
        const int key = k_lo + t * kTKT + r;
        return ((static_cast<int64_t>(page) * p.Hkv + kvh) << p.ps_log2) + (key & ps_mask);
      };
      constexpr int CPR = C::KROW / 16;  // 16-byte chunks per code row
#pragma unroll
      for (int h = 0; h < (kTKT * CPR) / kPThreads; ++h) {
        const int c = tid + h * kPThreads, r = c / CPR, cc = c - r * CPR;
        const int64_t row = row_of(r);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(base + c * 16),
                     "l"(p.kc + row * C::KROW + 16 * cc) : "memory");
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(base + kTKT * C::KROW + c * 16),
                     "l"(p.vc + row * C::KROW + 16 * cc) : "memory");
      }
      {  // scale rows: 16-byte chunk q of the tile's K (threads 0..) and V (threads 32..) scale rows
        constexpr int SCH = kTKT * C::SROW / 16;  // chunks per scale array
        const int q = tid & 31, is_v = tid >> 5;
        const int r = q * 16 / C::SROW;  // first key row of the chunk (a chunk never spans runs)
        const int64_t row = row_of(r < kTKT ? r : 0);
        if (q < SCH && is_v < 2)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(base + 2 * kTKT * C::KROW + is_v * (kTKT * C::SROW) + q * 16),
                       "l"((is_v ? p.vs : p.ks) + row * C::SROW) : "memory");
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&bars[st])) : "memory");
    };
    for (int t = 0; t < (ntiles < kTNST ? ntiles : kTNST); ++t) issue(t, page_of(t));
    // this thread's query row: the rotated E4M3 bytes, 16 per chunk, in the
    // swizzled K-major A layout of the block-scaled MMA
    {
      const uint8_t* qsrc = p.qbytes + ((static_cast<int64_t>(q0) + (my_row < nrows ? my_row / p.G : 0)) * p.Hq +
                                        kvh * p.G + (my_row < nrows ? my_row % p.G : 0)) * D;
#pragma unroll
      for (int ch = 0; ch < D / 16; ++ch) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (my_row < nrows) w = *reinterpret_cast<const uint4*>(qsrc + 16 * ch);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(q_u32 + tid * 128 + ((ch ^ (tid & 7)) << 4)),
                     "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w) : "memory");
      }
    }

    float m = -INFINITY, l = 0.f;
    float O[D];
#pragma unroll
    for (int k = 0; k < D; ++k) O[k] = 0.f;
    int RV = 0, badpos = 0x7FFFFFFF, win = 0;

    for (int t = 0; t < ntiles; ++t) {
      // page of the tile this iteration refills, loaded now so its latency hides behind the tile's work
      const int nxt_page = t + kTNST < ntiles ? page_of(t + kTNST) : 0;
      const int st = (git + t) % kTNST;
      const uint8_t* rk = raw + st * C::RAW;
      const uint8_t* rv = rk + kTKT * C::KROW;
      const uint8_t* rks = rv + kTKT * C::KROW;
      const uint8_t* rvs = rks + kTKT * C::SROW;
      const int kbase = k_lo + t * kTKT;
      const int slot = t & 1;
      // (a) the previous tile's P.V must be done before its operands are overwritten
      bool ok = true;
      if (pv_pending) {
        ok = mbar_spin(&bars[kTNST + 1], pv_phase & 1, kWaitBudget);
        ++pv_phase;
        pv_pending = false;
        tc_after();
      }
      ok = ok && mbar_spin(&bars[st], ((git + t) / kTNST) & 1, kWaitBudget);
      // (b) per key: the tile's largest V byte and first non-finite key
      if (tid < kTKT) {  // warps 0, 1: one key per thread, reduced per warp
        const int key = kbase + tid;
        int vmax = 0, bad = 0;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const int kb = rks[tid * C::SROW + g], vb = rvs[tid * C::SROW + g];
          if (vb != 0xFF) vmax = max(vmax, vb);  // a non-finite group is handled by badpos
          bad |= (kb == 0xFF) | (vb == 0xFF);
        }
        const bool in = key < k_hi;
        const unsigned wv = __reduce_max_sync(kFull, in ? static_cast<unsigned>(vmax) : 0u);
        const unsigned wb = __reduce_min_sync(kFull, (in && bad) ? static_cast<unsigned>(key) : 0x7FFFFFFFu);
        if (lane == 0) {  // this tile's slot, read by every thread below before its next write (tile t + 2)
          s_vmax[2 * slot + warp] = static_cast<int>(wv);
          s_bad[2 * slot + warp] = static_cast<int>(wb);
        }
      }
      if (__syncthreads_or(!ok)) {
        failed = true;
        break;
      }
      const int RVn = max(RV, max(s_vmax[2 * slot], s_vmax[2 * slot + 1]));
      badpos = min(badpos, min(s_bad[2 * slot], s_bad[2 * slot + 1]));
      // (c) K: the codes as they are, repacked from the cache's group-interleaved
      // words into the padded 4-bit operand layout (16 codes of natural channel
      // order in the first 8 bytes of each swizzled 16-byte chunk), and each key's
      // scale-byte word to tensor memory (key 32 j + i: lane i of every quarter,
      // column kSfbCol + j); V' = code * 2^(byte - RVn) (0 past the range), 8
      // channels of one key per thread and step.
#pragma unroll
      for (int h = 0; h < (kTKT * (D / 16)) / kPThreads; ++h) {
        const int c = tid + h * kPThreads;
        const int key = c / (D / 16), j = c - key * (D / 16);  // chunk j: natural words 2j, 2j+1
        const uint32_t* kw = reinterpret_cast<const uint32_t*>(rk + key * C::KROW);
        const uint32_t w0 = kw[NG * ((2 * j) & 3) + ((2 * j) >> 2)];
        const uint32_t w1 = kw[NG * ((2 * j + 1) & 3) + ((2 * j + 1) >> 2)];
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %3};" ::"r"(k_u32 + key * 128 + ((j ^ (key & 7)) << 4)),
                     "r"(w0), "r"(w1), "r"(0u) : "memory");
      }
      {
        uint32_t sf0, sf1;
        if (NG == 4) {
          sf0 = *reinterpret_cast<const uint32_t*>(rks + lane * 4);
          sf1 = *reinterpret_cast<const uint32_t*>(rks + (32 + lane) * 4);
        } else {
          sf0 = *reinterpret_cast<const uint16_t*>(rks + lane * 2);
          sf1 = *reinterpret_cast<const uint16_t*>(rks + (32 + lane) * 2);
        }
        asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(tmem + lanes + kSfbCol), "r"(sf0),
                     "r"(sf1) : "memory");
      }
      convert_v_half_row<D>(rv, rvs, tid, kbase + (tid >> 1) < k_hi, RVn, v_u32);
      tmem_wait_st();
      fence_proxy_async();  // generic-proxy operand writes, read next by the tensor cores
      tc_before();
      __syncthreads();
      // (d) S = Q K^T into tensor memory columns [0, 64): one block-scaled MMA per
      // 32-channel group, E4M3 query x E2M1 codes with the keys' UE8M0 bytes
      if (tid == 0) {
        tc_after();
#pragma unroll
        for (int g = 0; g < NG; ++g)
          tc_mma_bs(tmem, tc_desc(q_u32 + 32 * g), tc_desc(k_u32 + 32 * g), tc_idesc_bs(kTKT, g), tmem + kSfaCol,
                    tmem + kSfbCol, g > 0 ? 1u : 0u);
        tc_commit(&bars[kTNST]);
      }
      if (t + kTNST < ntiles) issue(t + kTNST, nxt_page);  // the raw stage is free again
      ok = mbar_spin(&bars[kTNST], s_phase & 1, kWaitBudget);
      ++s_phase;
      tc_after();
      // (e) this thread's row: logits, mask, online softmax, P to tensor memory
      float x[kTKT];
      {  // both halves of the row's logits in flight, one wait
        uint32_t ra[32], rb[32];
        tmem_ld32(tmem + lanes + 0, ra);
        tmem_ld32(tmem + lanes + 32, rb);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          x[k] = __uint_as_float(ra[k]);
          x[32 + k] = __uint_as_float(rb[k]);
        }
      }
      // x stays in the MMA's units; the softmax scale (> 0) is applied to the
      // maximum and fused into the exponent's argument below
      float mx = -INFINITY;
      if (kbase + kTKT <= k_hi && kbase + kTKT - 1 <= pos_lo && pos >= 0) {  // every key visible to the row
#pragma unroll
        for (int k = 0; k < kTKT; ++k) mx = fmaxf(mx, x[k]);
      } else {
#pragma unroll
        for (int k = 0; k < kTKT; ++k) {
          const int key = kbase + k;
          x[k] = (key <= pos && key < k_hi) ? x[k] : -INFINITY;
          mx = fmaxf(mx, x[k]);
        }
      }
      // the scale comes from shared memory once per tile: held in a register
      // across the whole kernel it costs the compiler spills of O
      float sl2e;
      asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sl2e) : "r"(smem_u32(s_sl2e)));
      mx *= sl2e;
      const bool need = mx > m + kTSlack || (m == -INFINITY && mx > -INFINITY);
      const bool fold = __syncthreads_or(need || !ok) != 0 || RVn != RV || win == kTWin;
      if (__syncthreads_or(!ok)) {
        failed = true;
        break;
      }
      if (fold) {
        if (win > 0) {  // the window's P.V finished in (a); add it to O with IEEE rounding
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r32[32];
            tmem_ld32(tmem + lanes + 128 + c0, r32);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) O[c0 + k] += __uint_as_float(r32[k]);
          }
        }
        if (need) {
          const float mn = fmaxf(m, mx);
          const float a = m == -INFINITY ? 0.f : ex2(m - mn);
#pragma unroll
          for (int k = 0; k < D; ++k) O[k] *= a;
          l *= a;
          m = mn;
        }
        if (RVn != RV) {
          const float f = pow2f(RV - RVn);
#pragma unroll
          for (int k = 0; k < D; ++k) O[k] *= f;
          RV = RVn;
        }
        win = 0;
      }
      {
        const float base = m == -INFINITY ? 0.f : m;
        uint32_t ph[32], pl[32];
#pragma unroll
        for (int k = 0; k < kTKT; k += 2) {
          const float p0 = ex2(fmaf(x[k], sl2e, -base)), p1 = ex2(fmaf(x[k + 1], sl2e, -base));
          l += p0 + p1;
          const float h0 = __uint_as_float(__float_as_uint(p0) & 0xFFFFE000u);
          const float h1 = __uint_as_float(__float_as_uint(p1) & 0xFFFFE000u);
          ph[k / 2] = pack_f16x2(h0, h1);
          pl[k / 2] = pack_f16x2(p0 - h0, p1 - h1);
        }
        tmem_st32(tmem + lanes + 0, ph);   // over this row's S, already read
        tmem_st32(tmem + lanes + 32, pl);
        tmem_wait_st();
      }
      tc_before();
      __syncthreads();
      // (f) O_win (+)= P V' into tensor memory columns [128, 128 + D)
      if (tid == 0) {
        tc_after();
#pragma unroll
        for (int j = 0; j < kTKT / 16; ++j) {  // keys 16 j .. 16 j + 15: two 8-key rows of swizzle atoms
          const uint64_t bd = tc_desc_mn(v_u32 + j * 2048, kTKT * 128);
          tc_mma_ts(tmem + 128, tmem + 8 * j, bd, tc_idesc(D, true), (win > 0 || j > 0) ? 1u : 0u);
          tc_mma_ts(tmem + 128, tmem + 32 + 8 * j, bd, tc_idesc(D, true), 1u);
        }
        tc_commit(&bars[kTNST + 1]);
      }
      pv_pending = true;
      ++win;
    }
    git += ntiles;
    if (failed) break;
    // the item's last window, then the partial (m, l, O) of this row
    bool ok = true;
    if (pv_pending) {
      ok = mbar_spin(&bars[kTNST + 1], pv_phase & 1, kWaitBudget);
      ++pv_phase;
      pv_pending = false;
      tc_after();
    }
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    if (win > 0) {
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t r32[32];
        tmem_ld32(tmem + lanes + 128 + c0, r32);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) O[c0 + k] += __uint_as_float(r32[k]);
      }
    }
    const float osc = pow2f(RV - 127);  // V' was code * 2^(byte - RV)
    ml_out[2 * tid] = m;
    ml_out[2 * tid + 1] = pos >= badpos ? __int_as_float(0x7FC00000) : l;
#pragma unroll
    for (int k = 0; k < D; k += 4)
      *reinterpret_cast<float4*>(o_out + static_cast<int64_t>(tid) * D + k) =
          make_float4(O[k] * osc, O[k + 1] * osc, O[k + 2] * osc, O[k + 3] * osc);
    tc_before();
    __syncthreads();  // every thread's tensor-memory reads done before the next item's MMAs
    tc_after();
  }
  if (failed) {
    if (tid == 0) {
      record_error(p.status, kErrTimeout);
      // let the MMAs in flight finish before the block's memory goes away
      if (pv_pending) mbar_wait(&bars[kTNST + 1], pv_phase & 1, kWaitBudget);
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // this thread's copies in flight land first
  tc_before();
  __syncthreads();
  if (warp == 0) {
    tc_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTCols));
  }
  pdl_trigger();
}

// ------------------------------------------------------------ warp-specialised variant (head_dim 128)
// The same items, arithmetic and partials as prefill_tc_kernel, with the
// tile's phases on separate warps so that they overlap across tiles:
//   * warp 8 fills a 4-stage raw ring with per-lane 16-byte cp.async (page
//     numbers one tile ahead);
//   * warps 4-7 ("convert"): the tile's V statistics, the K codes repacked into
//     the padded operand, the keys' scale words to tensor memory, V' in f16
//     (operands double-buffered), and per row (thread = row) the fp32 output
//     O, kept in tensor memory: each window of P.V sums is folded into O with
//     IEEE adds when the softmax warps ask for it, and O is written at the
//     item end;
//   * warps 0-3 ("softmax", thread = row): the item's query rows, then per
//     tile the row's logits from tensor memory, the mask, the lazy running
//     maximum (a window is closed, by the fold above, whenever any row's
//     maximum or the V reference grows, and every kTWin tiles) and P as hi + lo
//     f16 parts into tensor memory (S and P double-buffered);
//   * warp 9 (one thread) issues each tile's QK^T as soon as its operands are
//     ready, warp 10 (one thread) its P.V as soon as P is (tcgen05.mma holds its
//     issuing thread for about its execution time, so each MMA stream gets a
//     warp of its own; the registers are budgeted for 12 warps either way).
// Tensor memory: S/P [2][64] at 0, O_win at 128, query scale factors at 256,
// key scale factors [2] at 288 and 320, the folded fp32 output O at 384.
constexpr int kWThreads = 352;
constexpr int kWNst = 4;
constexpr uint32_t kWColO = 128, kWColSfa = 256, kWColSfb = 288, kWColAcc = 384;
constexpr int kWCols = 512;

struct WS {
  static constexpr int D = 128, KROW = 64, SROW = 4, NG = 4;
  static constexpr int RAW = 2 * kTKT * KROW + 2 * kTKT * SROW;  // 8704
  static constexpr int QB = kTRows * 128;
  static constexpr int KB = kTKT * 128;
  static constexpr int VB = kTKT * 2 * D;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QB;       // [2]
  static constexpr int OFF_V = OFF_K + 2 * KB;   // [2]
  static constexpr int OFF_RAW = OFF_V + 2 * VB; // [kWNst]
  static constexpr int OFF_MISC = OFF_RAW + kWNst * RAW;
  static constexpr int MISC = 4096;
  static constexpr int SMEM = OFF_MISC + MISC + 1024;
};
// barriers
enum WBar {
  kWFull = 0, kWEmpty = kWFull + kWNst, kWKv = kWEmpty + kWNst, kWS = kWKv + 2, kWP = kWS + 2, kWO = kWP + 2,
  kWFold = kWO + 2, kWQ = kWFold + 2, kWDone = kWQ + 1, kWBarCount = kWDone + 1
};
// misc byte offsets
constexpr int kWMTslot = 256, kWMAbort = 260, kWMSl2e = 264;
constexpr int kWMVmax = 384;          // [2 tiles][2 warps] int
constexpr int kWMBad = 400;           // [2 tiles][2 warps] int
constexpr int kWMRv = 288;            // [2] int: RVn of the tile
constexpr int kWMFl = 296;            // [2] int: fold flag of the tile
constexpr int kWMRvf = 304;           // [2] float: O's factor for a grown V reference
constexpr int kWMGfl = 320;           // [2][4] int
constexpr int kWMAlpha = 512;         // [2][128] float
constexpr int kWMMfin = kWMAlpha + 1024;  // [128] float
constexpr int kWMLfin = kWMMfin + 512;    // [128] float
static_assert(kWMLfin + 512 <= WS::MISC, "misc");

// the per-item quantities every role needs (as prefill_tc_kernel computes them)
struct WItem {
  int b, q0, n, nrows, L, ctx, kvh, row0, pos_lo, k_lo, k_hi, ntiles, lp_last;
  const int32_t* bt_row;
};
__device__ __forceinline__ WItem w_item(const PrefillParams& p, int64_t item, int splits, int kchunk, int cap,
                                        bool report) {
  WItem it;
  int lb = 1, hb = p.B;
  while (lb < hb) {
    const int mid = (lb + hb) >> 1;
    if (p.item_pre[mid] > item) hb = mid; else lb = mid + 1;
  }
  const int b = lb - 1;
  const int q0 = p.cu_q[b], n_plan = max(0, p.cu_q[b + 1] - q0);
  int L = p.seq_lens[b];
  int n = n_plan;
  if (p.cascade) {
    L = casc_shared_keys(n_plan, p.G, L, p.min_rows, p.casc_cap);
    if (q0 < 0 || q0 + n > p.T) {
      if (report) record_error(p.status, kErrBounds);
      L = 0;
    }
  } else if (L < 0 || L > cap || n > L || q0 < 0 || q0 + n > p.T) {
    if (report) record_error(p.status, kErrBounds);
    L = L < 0 ? 0 : (L > cap ? cap : L);
    n = n > L ? L : n;
    if (q0 < 0 || q0 + n > p.T) n = 0;
  }
  const int ctx = p.cascade ? 0 : L - n;
  const int tiles_b = row_tiles(n_plan, p.G, kTRows);
  const int64_t local = item - p.item_pre[b];
  const int kvh = static_cast<int>(local / (static_cast<int64_t>(tiles_b) * splits));
  const int rem = static_cast<int>(local - static_cast<int64_t>(kvh) * tiles_b * splits);
  const int rtile = rem / splits, split = rem - rtile * splits;
  const int row0 = rtile * kTRows, nrows = n * p.G;
  const int last_row = min(row0 + kTRows, nrows) - 1;
  const int pos_max = p.cascade ? L - 1 : ctx + last_row / p.G;
  it.b = b;
  it.q0 = q0;
  it.n = n;
  it.nrows = nrows;
  it.L = L;
  it.ctx = ctx;
  it.kvh = kvh;
  it.row0 = row0;
  it.pos_lo = p.cascade ? L - 1 : ctx + row0 / p.G;
  it.k_lo = split * kchunk;
  it.k_hi = min(it.k_lo + kchunk, pos_max + 1);
  it.ntiles = it.k_lo < it.k_hi ? (it.k_hi - it.k_lo + kTKT - 1) / kTKT : 0;
  it.lp_last = (L - 1) >> p.ps_log2;
  it.bt_row = p.block_table + static_cast<int64_t>(p.cascade ? q0 : b) * p.max_pages;
  return it;
}

__device__ __forceinline__ void w_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void w_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool w_poll(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok)
               : "r"(smem_u32(bar)), "r"(parity)
               : "memory");
  return ok != 0;
}
// Bounded wait; once any thread has timed out, every wait returns at once so
// that all roles run to the end with the same control flow.
__device__ __forceinline__ void w_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, unsigned int* status) {
  if (w_poll(bar, parity)) return;
  const long long t0 = clock64();
  while (!*abort_flag) {
    __nanosleep(32);
    if (w_poll(bar, parity)) return;
    if (clock64() - t0 > kWaitBudget) {
      record_error(status, kErrTimeout);
      *abort_flag = 1;
      return;
    }
  }
}

__global__ void __launch_bounds__(kWThreads, 1) prefill_ws_kernel(const __grid_constant__ PrefillParams p) {
  using C = WS;
  constexpr int D = C::D, NG = C::NG;
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  const uint32_t q_u32 = sb + C::OFF_Q, k_u32 = sb + C::OFF_K, v_u32 = sb + C::OFF_V;
  uint8_t* raw = sm + C::OFF_RAW;
  uint8_t* misc = sm + C::OFF_MISC;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(misc + kWMTslot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + kWMAbort);
  float* s_sl2e = reinterpret_cast<float*>(misc + kWMSl2e);
  int* s_vmax = reinterpret_cast<int*>(misc + kWMVmax);
  int* s_bad = reinterpret_cast<int*>(misc + kWMBad);
  int* s_rv = reinterpret_cast<int*>(misc + kWMRv);
  int* s_fl = reinterpret_cast<int*>(misc + kWMFl);
  float* s_rvf = reinterpret_cast<float*>(misc + kWMRvf);
  int* s_gfl = reinterpret_cast<int*>(misc + kWMGfl);
  float* s_alpha = reinterpret_cast<float*>(misc + kWMAlpha);
  float* s_mfin = reinterpret_cast<float*>(misc + kWMMfin);
  float* s_lfin = reinterpret_cast<float*>(misc + kWMLfin);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kWNst; ++s) {
      mbar_init(&bars[kWFull + s], 32);
      mbar_init(&bars[kWEmpty + s], 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kWKv + s], 4);
      mbar_init(&bars[kWS + s], 1);
      mbar_init(&bars[kWP + s], 4);
      mbar_init(&bars[kWO + s], 1);
      mbar_init(&bars[kWFold + s], 4);
    }
    mbar_init(&bars[kWQ], 4);
    mbar_init(&bars[kWDone], 2);
    fence_mbar_init();
    *abort_flag = 0;
    *s_sl2e = p.sl2e;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(kWCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = *tslot;
  if (warp < 4) {  // query scale factors: byte 127 (scale 1) for every row and group
    const uint32_t one = 0x7F7F7F7Fu;
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %1, %1, %1};" ::"r"(
                     tmem + (static_cast<uint32_t>(warp * 32) << 16) + kWColSfa),
                 "r"(one) : "memory");
    tmem_wait_st();
  }
  pdl_wait();
  int64_t total = p.item_pre[p.B];
  const int splits = p.item_pre[p.B + 1], kchunk = p.item_pre[p.B + 2];
  if (total > p.max_items || splits < 1 || kchunk < kTKT) {
    if (blockIdx.x == 0 && tid == 0) record_error(p.status, kErrBounds);
    total = 0;
  }
  const int cap = p.max_pages << p.ps_log2;
  tc_before();
  __syncthreads();
  tc_after();

  if (warp == 8) {
    // ------------------------------------------------------------ copy warp
    const int rows_per = min(1 << p.ps_log2, kTKT);
    const int rp_log2 = p.ps_log2 < 6 ? p.ps_log2 : 6;
    const int ps_mask = (1 << p.ps_log2) - 1;
    uint32_t g = 0;  // tiles issued so far
    for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
      const WItem it = w_item(p, item, splits, kchunk, cap, false);
      if (it.ntiles == 0) continue;
      auto page_of = [&](int t) {  // lane r: the page of run r of tile t
        int page = 0;
        if (lane < kTKT / rows_per && t < it.ntiles) {
          int lp = (it.k_lo + t * kTKT + lane * rows_per) >> p.ps_log2;
          lp = lp > it.lp_last ? it.lp_last : lp;
          page = it.bt_row[lp];
        }
        return page;
      };
      int pg = page_of(0);
      for (int t = 0; t < it.ntiles; ++t, ++g) {
        const int pg_next = page_of(t + 1);
        const int st = static_cast<int>(g % kWNst);
        if (g >= kWNst) w_wait(&bars[kWEmpty + st], ((g - kWNst) / kWNst) & 1, abort_flag, p.status);
        const uint32_t base = smem_u32(raw + st * C::RAW);
        auto row_of = [&](int r) {
          int page = __shfl_sync(kFull, pg, r >> rp_log2);
          if (page < 0 || page >= p.num_pages) {
            record_error(p.status, kErrBounds);
            page = 0;
          }
          const int key = it.k_lo + t * kTKT + r;
          return ((static_cast<int64_t>(page) * p.Hkv + it.kvh) << p.ps_log2) + (key & ps_mask);
        };
#pragma unroll
        for (int h = 0; h < (kTKT * 4) / 32; ++h) {  // code chunks: 4 per 64-byte row
          const int c = lane + 32 * h, r = c >> 2, cc = c & 3;
          const int64_t row = row_of(r);
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(base + c * 16),
                       "l"(p.kc + row * C::KROW + 16 * cc) : "memory");
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(base + kTKT * C::KROW + c * 16),
                       "l"(p.vc + row * C::KROW + 16 * cc) : "memory");
        }
        {  // scale rows: lanes 0-15 the K chunks, 16-31 the V chunks (4 keys each)
          const int q = lane & 15, is_v = lane >> 4;
          const int64_t row = row_of(q * 4);
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(base + 2 * kTKT * C::KROW + is_v * (kTKT * C::SROW) + q * 16),
                       "l"((is_v ? p.vs : p.ks) + row * C::SROW) : "memory");
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&bars[kWFull + st])) : "memory");
        pg = pg_next;
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 9) {
    // ------------------------------------------------------------ QK^T thread
    if (lane == 0) {
      // QK^T(g) once tile g's operands are written (which the convert warps do
      // only after P.V(g - 2) completed, so the S buffer it overwrites is free)
      // and, at an item's first tile, the item's query rows are staged
      uint32_t g = 0, items_q = 0;
      for (int64_t item = blockIdx.x; item < total && !*abort_flag; item += gridDim.x) {
        const WItem it = w_item(p, item, splits, kchunk, cap, false);
        if (it.ntiles == 0) continue;
        w_wait(&bars[kWQ], items_q & 1, abort_flag, p.status);
        ++items_q;
        for (int t = 0; t < it.ntiles; ++t, ++g) {
          w_wait(&bars[kWKv + (g & 1)], (g >> 1) & 1, abort_flag, p.status);
          tc_after();
          const uint32_t kt = k_u32 + (g & 1) * C::KB;
#pragma unroll
          for (int gg = 0; gg < NG; ++gg)
            tc_mma_bs(tmem + 64u * (g & 1), tc_desc(q_u32 + 32 * gg), tc_desc(kt + 32 * gg), tc_idesc_bs(kTKT, gg),
                      tmem + kWColSfa, tmem + kWColSfb + 32u * (g & 1), gg > 0 ? 1u : 0u);
          tc_commit(&bars[kWS + (g & 1)]);
        }
      }
      tc_commit(&bars[kWDone]);
      // this thread's MMAs in flight finish before the tensor memory is freed,
      // after an abort too (bounded, whatever the abort flag says)
      if (!mbar_wait_sleep(&bars[kWDone], 0, kWaitBudget)) record_error(p.status, kErrTimeout);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ P.V thread
    if (lane == 0) {
      // P.V(g) once P(g) is written and, when it opens a window, the closing
      // window has been folded
      uint32_t g = 0;
      uint32_t fcnt[2] = {0u, 0u};  // folds waited for, per tile parity
      for (int64_t item = blockIdx.x; item < total && !*abort_flag; item += gridDim.x) {
        const WItem it = w_item(p, item, splits, kchunk, cap, false);
        for (int t = 0; t < it.ntiles; ++t, ++g) {
          w_wait(&bars[kWP + (g & 1)], (g >> 1) & 1, abort_flag, p.status);
          const int fl = *reinterpret_cast<volatile int*>(&s_fl[g & 1]);
          if (fl) {
            w_wait(&bars[kWFold + (g & 1)], fcnt[g & 1] & 1, abort_flag, p.status);
            ++fcnt[g & 1];
          }
          tc_after();
          const uint32_t vt = v_u32 + (g & 1) * C::VB;
          const uint32_t pcol = tmem + 64u * (g & 1);
#pragma unroll
          for (int j = 0; j < kTKT / 16; ++j) {
            const uint64_t bd = tc_desc_mn(vt + j * 2048, kTKT * 128);
            tc_mma_ts(tmem + kWColO, pcol + 8 * j, bd, tc_idesc(D, true), (!fl || j > 0) ? 1u : 0u);
            tc_mma_ts(tmem + kWColO, pcol + 32 + 8 * j, bd, tc_idesc(D, true), 1u);
          }
          tc_commit(&bars[kWO + (g & 1)]);
        }
      }
      tc_commit(&bars[kWDone]);
      // this thread's MMAs in flight finish before the tensor memory is freed,
      // after an abort too (bounded, whatever the abort flag says)
      if (!mbar_wait_sleep(&bars[kWDone], 0, kWaitBudget)) record_error(p.status, kErrTimeout);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax warps (thread = row)
    const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t g = 0, items_done = 0;
    for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
      const WItem it = w_item(p, item, splits, kchunk, cap, tid == 0);
      const int my_row = it.row0 + tid;
      const int pos = my_row < it.nrows ? (p.cascade ? it.L - 1 : it.ctx + my_row / p.G) : -1;
      if (it.ntiles == 0) {
        p.ws_ml[item * (kTRows * 2) + 2 * tid] = -INFINITY;
        p.ws_ml[item * (kTRows * 2) + 2 * tid + 1] = 0.f;
        continue;
      }
      {  // this row's rotated E4M3 query bytes, swizzled K-major A operand
        const uint8_t* qsrc = p.qbytes + ((static_cast<int64_t>(it.q0) + (my_row < it.nrows ? my_row / p.G : 0)) * p.Hq +
                                          it.kvh * p.G + (my_row < it.nrows ? my_row % p.G : 0)) * D;
#pragma unroll
        for (int ch = 0; ch < D / 16; ++ch) {
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (my_row < it.nrows) w = *reinterpret_cast<const uint4*>(qsrc + 16 * ch);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(q_u32 + tid * 128 + ((ch ^ (tid & 7)) << 4)),
                       "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w) : "memory");
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) w_arrive(&bars[kWQ]);
      }
      float m = -INFINITY, l = 0.f;
      int RV = 0, win = 0;
      for (int t = 0; t < it.ntiles; ++t, ++g) {
        const int kbase = it.k_lo + t * kTKT;
        w_wait(&bars[kWS + (g & 1)], (g >> 1) & 1, abort_flag, p.status);
        tc_after();
        float x[kTKT];
        {  // both halves of the row's logits in flight, one wait
          uint32_t ra[32], rb[32];
          tmem_ld32(tmem + lanes + 64u * (g & 1), ra);
          tmem_ld32(tmem + lanes + 64u * (g & 1) + 32, rb);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            x[k] = __uint_as_float(ra[k]);
            x[32 + k] = __uint_as_float(rb[k]);
          }
        }
        float mx = -INFINITY;
        if (kbase + kTKT <= it.k_hi && kbase + kTKT - 1 <= it.pos_lo && pos >= 0) {
#pragma unroll
          for (int k = 0; k < kTKT; ++k) mx = fmaxf(mx, x[k]);
        } else {
#pragma unroll
          for (int k = 0; k < kTKT; ++k) {
            const int key = kbase + k;
            x[k] = (key <= pos && key < it.k_hi) ? x[k] : -INFINITY;
            mx = fmaxf(mx, x[k]);
          }
        }
        float sl2e;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sl2e) : "r"(smem_u32(s_sl2e)));
        mx *= sl2e;
        const bool need = mx > m + kTSlack || (m == -INFINITY && mx > -INFINITY);
        const int rvn = *reinterpret_cast<volatile int*>(&s_rv[g & 1]);
        const unsigned vote = __ballot_sync(kFull, need);
        if (lane == 0) s_gfl[(g & 1) * 4 + warp] = vote != 0u;
        w_bar(1, 128);
        const int* gf = s_gfl + (g & 1) * 4;
        const bool fold = t == 0 || (gf[0] | gf[1] | gf[2] | gf[3]) || rvn != RV || win == kTWin;
        if (fold) {
          float a = 1.f;
          if (need) {
            const float mn = fmaxf(m, mx);
            a = m == -INFINITY ? 0.f : ex2(m - mn);
            l *= a;
            m = mn;
          }
          s_alpha[(g & 1) * kTRows + tid] = a;
          if (tid == 0) {
            s_fl[g & 1] = 1;
            s_rvf[g & 1] = t == 0 ? 1.f : pow2f(RV - rvn);
          }
          RV = rvn;
          win = 0;
        } else if (tid == 0) {
          s_fl[g & 1] = 0;
        }
        ++win;
        {
          const float base = m == -INFINITY ? 0.f : m;
          uint32_t ph[32], pl[32];
#pragma unroll
          for (int k = 0; k < kTKT; k += 2) {
            const float p0 = ex2(fmaf(x[k], sl2e, -base)), p1 = ex2(fmaf(x[k + 1], sl2e, -base));
            l += p0 + p1;
            const float h0 = __uint_as_float(__float_as_uint(p0) & 0xFFFFE000u);
            const float h1 = __uint_as_float(__float_as_uint(p1) & 0xFFFFE000u);
            ph[k / 2] = pack_f16x2(h0, h1);
            pl[k / 2] = pack_f16x2(p0 - h0, p1 - h1);
          }
          tmem_st32(tmem + lanes + 64u * (g & 1), ph);
          tmem_st32(tmem + lanes + 64u * (g & 1) + 32, pl);
          tmem_wait_st();
        }
        tc_before();
        __syncwarp();
        if (lane == 0) w_arrive(&bars[kWP + (g & 1)]);
      }
      s_mfin[tid] = m;
      s_lfin[tid] = l;
      w_bar(3, 256);  // the convert warps write the item's partials
      w_bar(4, 256);  // and have read these rows before the next item reuses them
      ++items_done;
    }
  } else {
    // ------------------------------------------------------------ convert warps (thread ct = row)
    const int ct = tid - 128, cw = warp - 4;
    const uint32_t lanes = static_cast<uint32_t>(cw * 32) << 16;
    uint32_t g = 0;
    for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
      const WItem it = w_item(p, item, splits, kchunk, cap, false);
      if (it.ntiles == 0) continue;
      const int my_row = it.row0 + ct;
      const int pos = my_row < it.nrows ? (p.cascade ? it.L - 1 : it.ctx + my_row / p.G) : -1;
      int RV = 0, badpos = 0x7FFFFFFF;
      bool ovalid = false;  // O (tensor memory, columns kWColAcc..) holds a folded window of this item
      // fold of tile gt (local t_local): wait for its P (the flag), then, if it
      // opens a window, add the closing window into O and rescale
      auto fold_check = [&](uint32_t gt, int t_local) {
        w_wait(&bars[kWP + (gt & 1)], (gt >> 1) & 1, abort_flag, p.status);
        if (!*reinterpret_cast<volatile int*>(&s_fl[gt & 1])) return;
        if (t_local > 0) {  // the window P.V(gt - 1) closed
          w_wait(&bars[kWO + ((gt - 1) & 1)], ((gt - 1) >> 1) & 1, abort_flag, p.status);
          tc_after();
          const float f = s_alpha[(gt & 1) * kTRows + ct] * s_rvf[gt & 1];
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t w32[32], o32[32];
            tmem_ld32(tmem + lanes + kWColO + c0, w32);
            if (ovalid) tmem_ld32(tmem + lanes + kWColAcc + c0, o32);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const float o = ovalid ? __uint_as_float(o32[k]) + __uint_as_float(w32[k]) : __uint_as_float(w32[k]);
              o32[k] = __float_as_uint(o * f);
            }
            tmem_st32(tmem + lanes + kWColAcc + c0, o32);
          }
          tmem_wait_st();
          ovalid = true;
        }
        tc_before();
        __syncwarp();
        if (lane == 0) w_arrive(&bars[kWFold + (gt & 1)]);
      };
      for (int t = 0; t < it.ntiles; ++t, ++g) {
        const int st = static_cast<int>(g % kWNst);
        const uint8_t* rk = raw + st * C::RAW;
        const uint8_t* rv = rk + kTKT * C::KROW;
        const uint8_t* rks = rv + kTKT * C::KROW;
        const uint8_t* rvs = rks + kTKT * C::SROW;
        const int kbase = it.k_lo + t * kTKT;
        const int slot = g & 1;
        w_wait(&bars[kWFull + st], (g / kWNst) & 1, abort_flag, p.status);
        if (ct < kTKT) {  // per key (convert warps 0, 1): the largest V byte and the first non-finite key
          const int key = kbase + ct;
          int vmax = 0, bad = 0;
#pragma unroll
          for (int gg = 0; gg < NG; ++gg) {
            const int kb = rks[ct * C::SROW + gg], vb = rvs[ct * C::SROW + gg];
            if (vb != 0xFF) vmax = max(vmax, vb);
            bad |= (kb == 0xFF) | (vb == 0xFF);
          }
          const bool in = key < it.k_hi;
          const unsigned wv = __reduce_max_sync(kFull, in ? static_cast<unsigned>(vmax) : 0u);
          const unsigned wb = __reduce_min_sync(kFull, (in && bad) ? static_cast<unsigned>(key) : 0x7FFFFFFFu);
          if (lane == 0) {  // this tile's slot, read below by every convert thread before the next write (tile g + 2)
            s_vmax[2 * slot + cw] = static_cast<int>(wv);
            s_bad[2 * slot + cw] = static_cast<int>(wb);
          }
        }
        w_bar(2, 128);
        const int RVn = max(RV, max(s_vmax[2 * slot], s_vmax[2 * slot + 1]));
        badpos = min(badpos, min(s_bad[2 * slot], s_bad[2 * slot + 1]));
        if (ct == 0) s_rv[slot] = RVn;
        RV = RVn;
        // the operand buffers of this slot were last read by tile g - 2's MMAs
        if (g >= 2) w_wait(&bars[kWO + slot], ((g - 2) >> 1) & 1, abort_flag, p.status);
        tc_after();
        const uint32_t kt_u32 = k_u32 + slot * C::KB, vt_u32 = v_u32 + slot * C::VB;
#pragma unroll
        for (int h = 0; h < (kTKT * (D / 16)) / 128; ++h) {
          const int c = ct + h * 128;
          const int key = c / (D / 16), j = c - key * (D / 16);
          const uint32_t* kw = reinterpret_cast<const uint32_t*>(rk + key * C::KROW);
          const uint32_t w0 = kw[NG * ((2 * j) & 3) + ((2 * j) >> 2)];
          const uint32_t w1 = kw[NG * ((2 * j + 1) & 3) + ((2 * j + 1) >> 2)];
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %3};" ::"r"(kt_u32 + key * 128 + ((j ^ (key & 7)) << 4)),
                       "r"(w0), "r"(w1), "r"(0u) : "memory");
        }
        {
          const uint32_t sf0 = *reinterpret_cast<const uint32_t*>(rks + lane * 4);
          const uint32_t sf1 = *reinterpret_cast<const uint32_t*>(rks + (32 + lane) * 4);
          asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(
                           tmem + lanes + kWColSfb + 32u * slot),
                       "r"(sf0), "r"(sf1) : "memory");
        }
        convert_v_half_row<D>(rv, rvs, ct, kbase + (ct >> 1) < it.k_hi, RVn, vt_u32);
        tmem_wait_st();
        fence_proxy_async();
        tc_before();
        __syncwarp();
        if (lane == 0) {
          w_arrive(&bars[kWKv + slot]);
          w_arrive(&bars[kWEmpty + st]);
        }
        if (t >= 1) fold_check(g - 1, t - 1);
      }
      // the item's last tile: its fold, then the last window into O
      const uint32_t gl = g - 1;
      fold_check(gl, it.ntiles - 1);
      w_wait(&bars[kWO + (gl & 1)], (gl >> 1) & 1, abort_flag, p.status);
      tc_after();
      w_bar(3, 256);  // the softmax warps' (m, l) of this item are in shared memory
      const float osc = pow2f(RV - 127);  // V' was code * 2^(byte - RV)
      float* ml_out = p.ws_ml + item * (kTRows * 2);
      float* o_out = p.ws_o + item * (static_cast<int64_t>(kTRows) * D);
      const bool live = !*abort_flag;
      if (live) {
        ml_out[2 * ct] = s_mfin[ct];
        ml_out[2 * ct + 1] = pos >= badpos ? __int_as_float(0x7FC00000) : s_lfin[ct];
      }
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {  // O + the last window, scaled, to the item's partial
        uint32_t w32[32], o32[32];
        tmem_ld32(tmem + lanes + kWColO + c0, w32);
        if (ovalid) tmem_ld32(tmem + lanes + kWColAcc + c0, o32);
        tmem_wait_ld();
        if (live) {
#pragma unroll
          for (int k = 0; k < 32; k += 4) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              v[e] = (ovalid ? __uint_as_float(o32[k + e]) + __uint_as_float(w32[k + e]) : __uint_as_float(w32[k + e])) * osc;
            *reinterpret_cast<float4*>(o_out + static_cast<int64_t>(ct) * D + c0 + k) = make_float4(v[0], v[1], v[2], v[3]);
          }
        }
      }
      tc_before();
      w_bar(4, 256);
    }
  }
  tc_before();
  __syncthreads();
  tc_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kWCols));
  pdl_trigger();
}

struct PrefillMergeParams {
  const float* ws_ml;
  const float* ws_o;
  const int32_t* item_pre;
  const int32_t* cu_q;
  const int32_t* seq_lens;
  int B, T, Hq, G, cap, rows;
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
  const int splits = p.item_pre[p.B + 1];
  if (q0 < 0 || q0 + n > p.T || p.item_pre[p.B] > p.max_items || splits < 1) n = 0;
  const int i = t - q0;
  float o[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) o[e] = 0.f;
  if (i >= 0 && i < n) {
    const int kvh = h / p.G, hl = h - kvh * p.G;
    const int rowi = i * p.G + hl, rtile = rowi / p.rows, rr = rowi - rtile * p.rows;
    const int64_t item0 = p.item_pre[b] + (static_cast<int64_t>(kvh) * row_tiles(n_plan, p.G, p.rows) + rtile) * splits;
    float Ms = -INFINITY, Ls = 0.f;
    if (splits <= kMergeOneRound) {
      // one round: lane s holds (m, l) of split s, and every lane loads its chunk of
      // all the splits' O rows before any is used (an empty split's row is never read
      // into the sum: its m is -inf)
      float m = -INFINITY, l = 0.f;
      if (lane < splits) {
        m = p.ws_ml[((item0 + lane) * p.rows + rr) * 2];
        l = p.ws_ml[((item0 + lane) * p.rows + rr) * 2 + 1];
      }
      float ov[kMergeOneRound][EPL];
#pragma unroll
      for (int j = 0; j < kMergeOneRound; ++j)
        if (j < splits) {
          const float* src = p.ws_o + ((item0 + j) * p.rows + rr) * D + lane * EPL;
#pragma unroll
          for (int e = 0; e < EPL; ++e) ov[j][e] = src[e];
        }
      Ms = m;
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) Ms = fmaxf(Ms, __shfl_xor_sync(kFull, Ms, k));
      const bool live = m != -INFINITY;
      const float w = live ? ex2(m - Ms) : 0.f;
      Ls = w * l;
      const unsigned mask = __ballot_sync(kFull, live);
#pragma unroll
      for (int j = 0; j < kMergeOneRound; ++j) {
        const float wj = __shfl_sync(kFull, w, j);
        if (j < splits && ((mask >> j) & 1u)) {
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[e] += wj * ov[j][e];
        }
      }
    } else {
      for (int s0 = 0; s0 < splits; s0 += 32) {
        const int s = s0 + lane;
        if (s < splits) Ms = fmaxf(Ms, p.ws_ml[((item0 + s) * p.rows + rr) * 2]);
      }
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) Ms = fmaxf(Ms, __shfl_xor_sync(kFull, Ms, k));
      for (int s0 = 0; s0 < splits; s0 += 32) {
        const int s = s0 + lane;
        float w = 0.f;
        bool live = false;
        if (s < splits) {
          const float m = p.ws_ml[((item0 + s) * p.rows + rr) * 2];
          live = m != -INFINITY;  // an empty split wrote no output row
          if (live) {
            w = ex2(m - Ms);
            Ls += w * p.ws_ml[((item0 + s) * p.rows + rr) * 2 + 1];
          }
        }
        const unsigned mask = __ballot_sync(kFull, live);
        const int cnt = min(32, splits - s0);
        for (int j = 0; j < cnt; ++j) {
          const float wj = __shfl_sync(kFull, w, j);
          if ((mask >> j) & 1u) {
            const float* src = p.ws_o + ((item0 + s0 + j) * p.rows + rr) * D + lane * EPL;
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[e] += wj * src[e];
          }
        }
      }
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) Ls += __shfl_xor_sync(kFull, Ls, k);
    const float inv = 1.f / Ls;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] *= inv;
    inverse_rotate_warp<D>(o, lane, p.sign.m);  // out = R^T o
  }
  float* dst = p.out + row * D + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; ++e) dst[e] = o[e];
}

}  // namespace

// ------------------------------------------------------------------ host
namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace bound of one launch.  The split count itself is chosen on the
// device from the key ranges present (prefill_plan_kernel); the host fixes its
// largest value, `splits`: the count that gives two waves of two blocks per SM
// at the bound on row tiles, times four for the prefill when the row tiles
// alone give fewer than two waves (room for the device's choice; with more,
// extra splits only add partials), as is for the cascade prefix (the decode's
// merge reads that count).
struct PrefillPlan {
  int splits;
  int64_t max_items;
  size_t off_pre, off_q, off_ml, off_o, total;
};

PrefillPlan plan_prefill(int T, int B, int hq, int hkv, int d, int max_keys, int sms, int rows, bool fixed) {
  PrefillPlan pl;
  const int G = hq / hkv;
  const int64_t tiles = (static_cast<int64_t>(T) * G + rows - 1) / rows + B;  // bound on row tiles per kv head
  const int64_t base = static_cast<int64_t>(hkv) * tiles;
  const int64_t target = 2LL * 2 * sms;  // two waves of two blocks per SM
  const int max_splits = std::max(1, (max_keys + kTKT - 1) / kTKT);
  const int64_t s0 = std::max<int64_t>(1, (target + base - 1) / base);
  pl.splits = static_cast<int>(std::min<int64_t>(max_splits, fixed || base >= target ? s0 : 4 * s0));
  pl.max_items = base * pl.splits;
  pl.off_pre = 256;
  pl.off_q = pl.off_pre + align256(static_cast<size_t>(B + 3) * 4);
  pl.off_ml = pl.off_q + align256(static_cast<size_t>(T) * hq * d);
  pl.off_o = pl.off_ml + align256(static_cast<size_t>(pl.max_items) * rows * 2 * 4);
  pl.total = pl.off_o + static_cast<size_t>(pl.max_items) * rows * d * 4;
  return pl;
}

constexpr int kItemRows = kTRows;  // query rows per work item

// Kernel attributes, once per device; the CTAs per SM.
template <int D>
int prefill_ctas_per_sm() {
  static std::mutex cfg_mu;
  static bool done[uqh::kMaxDevices];
  const uqh::DevInfo& di = uqh::dev_info();
  if (di.device < 0) return 0;
  {
    std::lock_guard<std::mutex> lk(cfg_mu);
    if (!done[di.device]) {
      if (cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC<D>::SMEM) !=
              cudaSuccess ||
          cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout, 100) !=
              cudaSuccess)
        return 0;
      done[di.device] = true;
    }
  }
  // Two CTAs per SM: their shared memory (2 x 93 KB), registers (2 x 128 x 255)
  // and tensor-memory columns (2 x 256 of 512) fit, and each CTA's serial phases
  // (convert, QK^T, softmax, P.V) overlap the other's.  The occupancy query
  // reports one for this kernel; measured, two are resident.
  return 512 / kTCols;
}

// Parameters common to prefill and the cascade prefix; the caller sets the rest.
template <int D>
PrefillParams base_params(const uq_cache& c, const int32_t* block_table, int max_pages, int B, int T, int hq,
                          float sm_scale, const PrefillPlan& pl, uint8_t* ws) {
  PrefillParams p;
  p.qbytes = ws + pl.off_q;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.kc = static_cast<const uint8_t*>(c.k_codes);
  p.ks = static_cast<const uint8_t*>(c.k_scales);
  p.vc = static_cast<const uint8_t*>(c.v_codes);
  p.vs = static_cast<const uint8_t*>(c.v_scales);
  p.B = B;
  p.T = T;
  p.Hq = hq;
  p.Hkv = c.num_kv_heads;
  p.G = hq / c.num_kv_heads;
  p.ps_log2 = uqh::ilog2(c.page_size);
  p.num_pages = c.num_pages;
  const float sm = sm_scale > 0.f ? sm_scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  p.sl2e = sm * 1.4426950408889634f;
  p.ws_ml = reinterpret_cast<float*>(ws + pl.off_ml);
  p.ws_o = reinterpret_cast<float*>(ws + pl.off_o);
  p.item_pre = reinterpret_cast<int32_t*>(ws + pl.off_pre);
  p.max_items = pl.max_items;
  p.status = uqh::status_word();
  p.cascade = 0;
  p.min_rows = 0;
  p.casc_cap = 0;
  return p;
}

// Head_dim 128 runs the warp-specialised kernel unless UQ_PREFILL=tc selects
// the single-role one (read once per process); head_dim 64 always runs the
// single-role kernel.
bool prefill_ws_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("UQ_PREFILL");
    return !(e != nullptr && std::strcmp(e, "tc") == 0);
  }();
  return on;
}

// CTAs of the item kernel's grid (0 on failure).

// One CTA per SM; the dynamic shared-memory attribute once per device.
int prefill_ws_ctas_per_sm() {
  static std::mutex cfg_mu;
  static bool done[uqh::kMaxDevices];
  const uqh::DevInfo& di = uqh::dev_info();
  if (di.device < 0) return 0;
  std::lock_guard<std::mutex> lk(cfg_mu);
  if (!done[di.device]) {
    if (cudaFuncSetAttribute(prefill_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, WS::SMEM) != cudaSuccess)
      return 0;
    done[di.device] = true;
  }
  return 1;
}

// CTAs of the item kernel's grid (0 on failure).
template <int D>
int item_grid(const PrefillPlan& pl) {
  const int per_sm = (D == 128 && prefill_ws_enabled()) ? prefill_ws_ctas_per_sm() : prefill_ctas_per_sm<D>();
  if (per_sm < 1) return 0;
  return static_cast<int>(std::max<int64_t>(
      1, std::min<int64_t>(pl.max_items, static_cast<int64_t>(uqh::dev_info().sms) * per_sm)));
}

template <int D>
uq_status launch_items(const PrefillParams& p, int grid, cudaStream_t s) {
  if (D == 128 && prefill_ws_enabled())
    return uqh::cuda_status(
        uqh::launch_pdl(prefill_ws_kernel, static_cast<unsigned>(grid), kWThreads, WS::SMEM, s, p));
  return uqh::cuda_status(
      uqh::launch_pdl(prefill_tc_kernel<D>, static_cast<unsigned>(grid), kPThreads, TC<D>::SMEM, s, p));
}

template <int D>
uq_status run_prefill(const uqh::PrefillArgs& a, cudaStream_t s) {
  const uq_cache& c = *a.cache;
  const int G = a.num_q_heads / c.num_kv_heads;
  const int cap = a.max_pages * c.page_size;
  const PrefillPlan pl = plan_prefill(a.num_q_tokens, a.batch, a.num_q_heads, c.num_kv_heads, D, cap,
                                      uqh::dev_info().sms, kItemRows, false);
  if (a.ws_bytes < pl.total) return UQ_ERR_WORKSPACE;
  const int grid = item_grid<D>(pl);
  if (grid < 1) return UQ_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  PrefillParams p = base_params<D>(c, a.block_table, a.max_pages, a.batch, a.num_q_tokens, a.num_q_heads,
                                   a.sm_scale, pl, ws);
  if (!p.status) return UQ_ERR_CUDA;
  p.cu_q = a.cu_q;
  p.seq_lens = a.seq_lens;
  prefill_plan_kernel<<<1, 32, 0, s>>>(a.cu_q, a.seq_lens, a.batch, G, c.num_kv_heads, pl.splits, 0, kItemRows,
                                       nullptr, 0, cap, grid, p.item_pre);
  if (cudaGetLastError() != cudaSuccess) return UQ_ERR_CUDA;
  uq_status st = uqh::launch_query_fp8(a.q, static_cast<int64_t>(a.num_q_tokens) * a.num_q_heads, D,
                                            c.rot_seed, ws + pl.off_q, s);
  if (st != UQ_OK) return st;
  st = launch_items<D>(p, grid, s);
  if (st != UQ_OK) return st;
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
  mp.rows = kItemRows;
  mp.max_items = pl.max_items;
  mp.cap = cap;
  mp.out = a.out;
  uqh::make_sign_masks(c.rot_seed, D, &mp.sign);
  const int64_t rows = static_cast<int64_t>(a.num_q_tokens) * a.num_q_heads;
  return uqh::cuda_status(
      uqh::launch_pdl(prefill_merge_kernel<D>, static_cast<unsigned>((rows + 3) / 4), 128, 0, s, mp));
}

template <int D>
uq_status run_cascade_prefix(const void* q, const uq_cache& c, const int32_t* block_table, int max_pages, int batch,
                             int hq, const uqh::CascadeGroups& cg, float sm_scale, void* ws_v, size_t ws_bytes,
                             uqh::PrefixPartials* out, cudaStream_t s) {
  const int G = hq / c.num_kv_heads;
  const PrefillPlan pl = plan_prefill(batch, cg.groups, hq, c.num_kv_heads, D, cg.cap, uqh::dev_info().sms,
                                      kItemRows, true);
  if (ws_bytes < pl.total) return UQ_ERR_WORKSPACE;
  const int grid = item_grid<D>(pl);
  if (grid < 1) return UQ_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(ws_v);
  PrefillParams p = base_params<D>(c, block_table, max_pages, cg.groups, batch, hq, sm_scale, pl, ws);
  if (!p.status) return UQ_ERR_CUDA;
  p.cu_q = cg.cu;
  p.seq_lens = cg.prefix;
  p.cascade = 1;
  p.min_rows = cg.min_rows;
  p.casc_cap = cg.cap;
  prefill_plan_kernel<<<1, 32, 0, s>>>(cg.cu, nullptr, cg.groups, G, c.num_kv_heads, pl.splits, pl.splits,
                                       kItemRows, cg.prefix, cg.min_rows, cg.cap, grid, p.item_pre);
  if (cudaGetLastError() != cudaSuccess) return UQ_ERR_CUDA;
  uq_status st = uqh::launch_query_fp8(q, static_cast<int64_t>(batch) * hq, D, c.rot_seed, ws + pl.off_q, s);
  if (st != UQ_OK) return st;
  st = launch_items<D>(p, grid, s);
  if (st != UQ_OK) return st;
  out->ml = p.ws_ml;
  out->o = p.ws_o;
  out->item_pre = p.item_pre;
  out->splits = pl.splits;
  out->rows = kItemRows;
  out->max_items = pl.max_items;
  return UQ_OK;
}

}  // namespace

namespace uqh {

size_t prefill_workspace_bytes(int T, int B, int hq, int hkv, int d, int max_keys) {
  return plan_prefill(T, B, hq, hkv, d, max_keys, std::max(1, dev_info().sms), kItemRows, false).total;
}

uq_status launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  return a.cache->head_dim == 128 ? run_prefill<128>(a, s) : run_prefill<64>(a, s);
}

size_t cascade_prefix_workspace_bytes(int batch, int groups, int hq, int hkv, int d, int max_keys) {
  return plan_prefill(batch, groups, hq, hkv, d, max_keys, std::max(1, dev_info().sms), kItemRows, true).total;
}

uq_status launch_cascade_prefix(const void* q, const uq_cache* cache, const int32_t* block_table, int32_t max_pages,
                                int32_t batch, int32_t num_q_heads, const CascadeGroups& cg, float sm_scale, void* ws,
                                size_t ws_bytes, PrefixPartials* out, cudaStream_t s) {
  return cache->head_dim == 128
             ? run_cascade_prefix<128>(q, *cache, block_table, max_pages, batch, num_q_heads, cg, sm_scale, ws,
                                       ws_bytes, out, s)
             : run_cascade_prefix<64>(q, *cache, block_table, max_pages, batch, num_q_heads, cg, sm_scale, ws,
                                      ws_bytes, out, s);
}

}  // namespace uqh
