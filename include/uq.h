/*
 * uq.h -- C ABI of libuq.so: a paged 4-bit KV cache (FP4 E2M1 codes with one
 * UE8M0 scale byte per 32 channels, "UltraQuant") for single-token decode
 * attention on NVIDIA GB300 (sm_103a), plus FP8-E4M3 and BF16 caches of the
 * same shape as comparison anchors.
 *
 * Sources of the operations (cited by page title and section):
 *   [UQ-review]    "UltraQuant: 4-bit KV Caching for Context-Heavy Agents",
 *                  review at manon006.tistory.com/395: §3.1 write path and
 *                  storage format, §3.2 dequantisation rule and FP8 query,
 *                  §3.3 constant c, §4.2 decode kernel (query rounded outside
 *                  the K-tile loop, cache layout matched to the scale operand).
 *   [UQ-residency] "kv-cache-4bit-serving-residency-collapse",
 *                  pheeree.github.io (2026-09-01): layout and dequant rule
 *                  (footnote 2), c ablation (footnote 13).
 *   [TQ-guide]     "TurboQuant 완전 정리" (juhoplayground.github.io):
 *                  randomised Hadamard rotation, orthogonality.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers unless a parameter says "host".
 *     The caller allocates and owns every buffer (cache, workspace, outputs);
 *     the library allocates no memory and keeps no state between calls other
 *     than one device status word per device (see uq_check_device_status).
 *   - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *     stream).  Argument checks happen synchronously, before anything is
 *     enqueued; a failed check enqueues nothing.
 *   - Every call returns a uq_status; no C++ exception crosses the ABI.
 *     UQ_ERR_CUDA means a CUDA runtime call or kernel launch failed.
 *   - Calls are thread-safe.  Calls that write the same cache region, or share
 *     a workspace, must be ordered by the caller (same stream or events).
 *   - Device-side range checks (slot, page, sequence length out of bounds) and
 *     bounded waits inside kernels never fault or hang: they record
 *     UQ_ERR_DEVICE_BOUNDS / UQ_ERR_DEVICE_TIMEOUT in the device status word,
 *     skip the offending access, and the host reads the word with
 *     uq_check_device_status.
 */
#ifndef UQ_H_
#define UQ_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum uq_status {
  UQ_OK = 0,
  UQ_ERR_INVALID_ARG = 1,    /* null pointer, negative size, inconsistent shapes */
  UQ_ERR_UNSUPPORTED = 2,    /* valid but unimplemented shape (head_dim, page size, batch) */
  UQ_ERR_ALIGNMENT = 3,      /* a pointer is not 16-byte aligned */
  UQ_ERR_WORKSPACE = 4,      /* workspace too small */
  UQ_ERR_CUDA = 5,           /* CUDA runtime / launch error */
  UQ_ERR_DEVICE_TIMEOUT = 6, /* a bounded wait inside a kernel ran out (device status word) */
  UQ_ERR_DEVICE_BOUNDS = 7   /* a slot / page / length index was out of range (device status word) */
} uq_status;

typedef enum uq_kv_dtype {
  UQ_FP4_UE8M0 = 0, /* rotated FP4 E2M1 codes + UE8M0 group scales, 4.25 bit/elem */
  UQ_FP8_E4M3 = 1,  /* unrotated E4M3 with one per-tensor scale for K and one for V */
  UQ_BF16 = 2,      /* unrotated bf16 */
  UQ_TQ4 = 3        /* rotated TurboQuant Q_mse: 4-bit Lloyd-Max codebook indices + fp32 row norm */
} uq_kv_dtype;

typedef enum uq_in_dtype { UQ_IN_BF16 = 0, UQ_IN_FP32 = 1 } uq_in_dtype;

/*
 * A paged KV cache.  All pointers are device pointers owned by the caller.
 * Physical rows are addressed [page][kv_head][offset] with page in
 * [0, num_pages), offset in [0, page_size); a token's slot is
 * page * page_size + offset (the vLLM convention).
 *
 *   UQ_FP4_UE8M0: k_codes, v_codes : uint8 [num_pages][num_kv_heads][page_size][head_dim/2]
 *                   codes of the ROTATED vector ([UQ-review] §3.1).  Natural
 *                   byte j of a row = code(2j) | code(2j+1) << 4, so group g
 *                   owns natural bytes 16g..16g+15 (words w = 0..3 of 4 bytes).
 *                   V rows are stored in natural order.  K rows are stored
 *                   group-interleaved by words: word w of group g sits at word
 *                   position (head_dim/32)*w + g, so every aligned run of
 *                   head_dim/8 bytes holds one word of each group (the layout
 *                   the decode consumes with one load per token; [UQ-review]
 *                   §4.2 matches the cache layout to the kernel's scale use);
 *                 k_scales, v_scales: uint8 [num_pages][num_kv_heads][page_size][head_dim/32]
 *                   UE8M0 byte of channels 32g..32g+31; value = code * 2^(byte-127)
 *                   ([UQ-review] §3.2); 0xFF marks a non-finite group.
 *                 17 bytes per 32 elements ([UQ-review] §3.1).
 *   UQ_FP8_E4M3:  k_codes, v_codes : uint8 [num_pages][num_kv_heads][page_size][head_dim],
 *                   element = e4m3(x / k_scale) (resp. v_scale); scales unused (NULL).
 *   UQ_BF16:      k_codes, v_codes : bf16  [num_pages][num_kv_heads][page_size][head_dim]; scales unused.
 *   UQ_TQ4:       the TurboQuant Q_mse codebook variant ([TQ-guide] "Lloyd-Max
 *                 스칼라 양자화 (Q_mse)"), a quality anchor for the FP4 format.
 *                 k_codes, v_codes : uint8, laid out exactly as for UQ_FP4_UE8M0
 *                   (K rows group-interleaved by words, V rows natural), each
 *                   nibble a sign-magnitude codebook index of one coordinate
 *                   of the ROTATED row divided by its norm: bit 3 = negative,
 *                   bits 0..2 = rank m of the magnitude, value = +-c_m with
 *                   c_0 < ... < c_7 the non-negative half of the 16-level
 *                   Lloyd-Max codebook of one coordinate of a random unit
 *                   vector in R^head_dim, stored as f16 (see uq_tq_codebook);
 *                 k_scales, v_scales: fp32 [num_pages][num_kv_heads][page_size]
 *                   the row's L2 norm n (NaN for a non-finite row, whose codes
 *                   are 0).  Element value = +-c_m * n.
 *                 4.25 bits per element at head_dim 128 (64 + 4 bytes per row).
 *
 * rot_seed seeds the ±1 diagonal of the randomised Hadamard rotation (FP4 and
 * TQ4); one sign vector serves K, V, the query and every head.  The same
 * seed must be used for append and decode.
 */
typedef struct uq_cache {
  int32_t dtype;        /* uq_kv_dtype */
  int32_t num_pages;
  int32_t num_kv_heads;
  int32_t page_size;    /* power of two, 16..256 */
  int32_t head_dim;     /* 64, 128 or 256 (TQ4: 64 or 128) */
  void* k_codes;
  void* k_scales;
  void* v_codes;
  void* v_scales;
  float k_scale;        /* FP8 only (1.0 if unused) */
  float v_scale;        /* FP8 only (1.0 if unused) */
  uint64_t rot_seed;    /* FP4 and TQ4 */
  float fp4_c;          /* FP4: the constant c of the scale rule, t = fl32(c * absmax); 0 selects
                           the pages' 0.156f ([UQ-review] §3.3).  A per-layer constant is the
                           pages' open option ([UQ-review] §7.3); uq_calibrate_c measures one.
                           Negative, NaN or infinite: UQ_ERR_INVALID_ARG. */
} uq_cache;

/* Byte size of array `which` of the cache (0 = k_codes, 1 = k_scales,
 * 2 = v_codes, 3 = v_scales); 0 for an unused array or invalid arguments.
 * Host-only; enqueues nothing. */
size_t uq_cache_bytes(const uq_cache* cache, int32_t which);

/*
 * Quantize-append ([UQ-review] §3.1 write path): for each token t with
 * slot_mapping[t] >= 0 and each kv head h, the rows k[t][h][:] and v[t][h][:]
 * are written into the cache at that slot.
 *   FP4:  y = fl32(FWHT_fp32(s .* x) * fl32(1/sqrt(head_dim))) (Walsh-Hadamard
 *         rotation, Sylvester order, stages in ascending stride), then per
 *         32-channel group m = max|y|, E = nearest integer to
 *         log2(fl32(0.156f * m)), byte = clamp(E + 127, 0, 254), codes =
 *         E2M1(y * 2^-E) rounded to nearest, ties to even, saturating at 6.
 *   FP8:  e4m3(x / k_scale), round to nearest even, saturating at 448.
 *   BF16: x rounded to bf16 (exact copy for bf16 input).
 *   TQ4:  y = the FP4 rotation of x; S = fp32 pairwise sum of fl32(y_i^2)
 *         (balanced binary tree over adjacent elements: left half + right
 *         half, recursively); n = fl32(sqrt(S)); with the codebook's fp32
 *         thresholds tau_0 < ... < tau_6 between c_0..c_7 and t_k =
 *         fl32(n * tau_k): y_i >= 0 gets code #{k : y_i >= t_k}, y_i < 0 gets
 *         8 | #{k : |y_i| > t_k} (the nearest codebook value of y_i / n,
 *         decided without a division).  A non-finite n stores NaN and zero
 *         codes.
 * k, v         : device, [num_tokens][num_kv_heads][head_dim], bf16 or fp32
 *                per in_dtype, 16-byte aligned rows (contiguous).
 * slot_mapping : device int64 [num_tokens]; negative = skip the token.
 *                Slots >= num_pages*page_size are skipped and recorded as
 *                UQ_ERR_DEVICE_BOUNDS.
 * block_table, max_pages_per_seq: accepted for interface symmetry with the
 *                decode call and unused (slots are physical); may be NULL/0.
 * num_tokens == 0 is a no-op.
 */
uq_status uq_quantize_append(const void* k, const void* v, int32_t in_dtype, int64_t num_tokens,
                             const int32_t* block_table, int32_t max_pages_per_seq,
                             const int64_t* slot_mapping, const uq_cache* cache,
                             cudaStream_t stream);

/* Workspace bytes that uq_decode_attention needs for this batch shape on the
 * current device.  Host-only.  A smaller workspace is accepted as long as it
 * holds at least one split per (sequence, kv head) plus one; the kernel then
 * uses fewer blocks. */
size_t uq_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim);

/*
 * Decode attention for one query token per sequence, straight from the
 * cache ([UQ-review] §3.2, §4.2):
 *   FP4:  q~ = e4m3(R q) (rotation as in append, then E4M3 round to nearest
 *         even, saturating; computed once per block, outside the page loop);
 *         logits_j = sm_scale * <q~, k^_j> with k^ = code * 2^(byte-127);
 *         softmax over j < seq_lens[b]; o = sum_j p_j v^_j; out = R^T o
 *         (inverse rotation; R is orthogonal, [TQ-guide]).
 *   FP8 / BF16: the same with q in bf16, k^ = e4m3 * k_scale (or bf16) and
 *         no rotation.
 * Query head h reads kv head h / (num_q_heads / num_kv_heads).
 * The key range is split over many blocks (split-K over 16-token chunks of
 * pages) and the partial results are merged with a log-sum-exp combine.
 * q           : device bf16 [batch][num_q_heads][head_dim]
 * block_table : device int32 [batch][max_pages_per_seq]; logical token j of
 *               sequence b lives in page block_table[b][j / page_size] at
 *               offset j % page_size.
 * seq_lens    : device int32 [batch]; 0 gives a zero output row.
 * sm_scale    : softmax scale; <= 0 selects 1/sqrt(head_dim).
 * out         : device fp32 [batch][num_q_heads][head_dim].
 * workspace   : device, >= 16-byte aligned, workspace_bytes long (see
 *               uq_decode_workspace_bytes); contents need not be initialised.
 * Supported: head_dim 64, 128 or 256 (TQ4: 64 or 128), page_size a power of
 * two in [16, 256], num_q_heads a multiple of num_kv_heads, batch <= 4096.
 */
uq_status uq_decode_attention(const void* q, const uq_cache* cache, const int32_t* block_table,
                              int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                              int32_t num_q_heads, float sm_scale, float* out, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/*
 * One decode step with the step's new tokens appended in the same launch
 * (FP4 cache only): for each sequence b with new_slots[b] >= 0, the token
 * k_new[b], v_new[b] is quantised exactly as uq_quantize_append would and
 * written to slot new_slots[b]; then the attention of uq_decode_attention is
 * computed over seq_lens[b] tokens, which include the new token as the last
 * one.  The pages describe the cache as written once per token and read by
 * the decode kernel ([UQ-review] §4.2); doing both in one launch saves the
 * separate append kernel of every decode step.
 * k_new, v_new : device [batch][num_kv_heads][head_dim], bf16 or fp32 as
 *                in_dtype says, 16-byte aligned.
 * new_slots    : device int64 [batch], 8-byte aligned; the physical slot of
 *                sequence b's new token, which must be where block_table
 *                places its logical position seq_lens[b] - 1 (a mismatch is
 *                recorded as UQ_ERR_DEVICE_BOUNDS and that token is not
 *                written); -1 = no new token (seq_lens[b] must then not
 *                count one).
 * Other arguments and errors as uq_decode_attention.  UQ_ERR_UNSUPPORTED for
 * FP8 / BF16 / TQ4 caches and for head_dim 256.
 */
uq_status uq_decode_attention_append(const void* q, const void* k_new, const void* v_new, int32_t in_dtype,
                                     const int64_t* new_slots, const uq_cache* cache, const int32_t* block_table,
                                     int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                                     int32_t num_q_heads, float sm_scale, float* out, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream);

/* The anchors: identical to uq_decode_attention but require cache->dtype to be
 * UQ_FP8_E4M3 (resp. UQ_BF16, UQ_TQ4) and return UQ_ERR_INVALID_ARG otherwise.
 * TQ4 ([TQ-guide] "직교성을 이용한 내적 보존"): q~ = f16(R q) (rotation as in
 * append, round to nearest even), logits_j = sm_scale * n^K_j * <q~, c(k_j)>,
 * softmax, o = sum_j p_j n^V_j c(v_j), out = R^T o; the codebook values
 * c(.) are the f16 values uq_tq_codebook returns. */
uq_status uq_decode_attention_fp8(const void* q, const uq_cache* cache, const int32_t* block_table,
                                  int32_t max_pages_per_seq, const int32_t* seq_lens,
                                  int32_t batch, int32_t num_q_heads, float sm_scale, float* out,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream);
uq_status uq_decode_attention_bf16(const void* q, const uq_cache* cache,
                                   const int32_t* block_table, int32_t max_pages_per_seq,
                                   const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                   float sm_scale, float* out, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream);
uq_status uq_decode_attention_tq4(const void* q, const uq_cache* cache, const int32_t* block_table,
                                  int32_t max_pages_per_seq, const int32_t* seq_lens,
                                  int32_t batch, int32_t num_q_heads, float sm_scale, float* out,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Chunked-prefill attention over an FP4 cache.  A prefill chunk first appends
 * its n_b new tokens of sequence b with uq_quantize_append; then query i of
 * the chunk (position p = seq_lens[b] - n_b + i) attends causally to keys
 * 0..p of the sequence, with the decode's numerics ([UQ-review] §3.2: rotated
 * E4M3 query, E2M1 x UE8M0 keys and values, fp32 output rotated back):
 * out[t][h] = R^T softmax_j(sm_scale <q~_t, k^_j>) v^_j over j <= p.
 * q           : device bf16 [num_q_tokens][num_q_heads][head_dim], 16-byte aligned;
 *               the chunk of sequence b is rows cu_q[b] .. cu_q[b+1]-1.
 * cu_q        : device int32 [batch + 1], non-decreasing, cu_q[0] = 0,
 *               cu_q[batch] = num_q_tokens.
 * seq_lens    : device int32 [batch]; keys of sequence b INCLUDING its chunk
 *               (n_b <= seq_lens[b]; a violation is recorded as
 *               UQ_ERR_DEVICE_BOUNDS and the chunk is clamped).
 * block_table, max_pages_per_seq, sm_scale: as uq_decode_attention.
 * out         : device fp32 [num_q_tokens][num_q_heads][head_dim].
 * workspace   : device, 16-byte aligned, at least
 *               uq_prefill_workspace_bytes(num_q_tokens, batch, num_q_heads,
 *               num_kv_heads, head_dim, max_pages_per_seq * page_size) bytes.
 *               The key ranges are split over work items on the device, from
 *               seq_lens (the longest sequence present, not the table's
 *               capacity); the workspace bounds the largest split count.
 * FP4 caches with head_dim 64 or 128 (UQ_ERR_UNSUPPORTED otherwise); other
 * shapes as the decode.
 */
size_t uq_prefill_workspace_bytes(int32_t num_q_tokens, int32_t batch, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t max_keys);
uq_status uq_prefill_attention(const void* q, const int32_t* cu_q, int32_t num_q_tokens, const uq_cache* cache,
                               const int32_t* block_table, int32_t max_pages_per_seq, const int32_t* seq_lens,
                               int32_t batch, int32_t num_q_heads, float sm_scale, float* out, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream);

/*
 * c calibration ([UQ-residency]: the shrink constant is the c minimising
 * E[(z - c m q(z / (c m)))^2] over rotated groups, z an element, m the group's
 * absolute maximum, q the E2M1 grid; [UQ-review] §7.3: per-layer constants).
 * Rotates n_vec rows x ([n_vec][head_dim], bf16 or fp32, device, 16-byte
 * aligned) with the cache rotation of rot_seed and, for each of the n_c
 * constants c_list[i] (host, 1 <= n_c <= 64, each finite > 0), writes to
 * sse[i] (device fp64 [n_c], 8-byte aligned; overwritten) the sum over all
 * elements of (z - rec)^2, where rec is the round trip of z through:
 *   mode  0: the deployed rule of uq_quantize_append with c = c_list[i]
 *            (UE8M0 byte of fl32(c m), E2M1 codes of z 2^-E);
 *   mode -1: a continuous scale s = c m (codes of fl32(z / s), rec = s value).
 * Groups with m = 0 add nothing; a non-finite group makes sse[i] NaN.  Set a
 * layer's uq_cache.fp4_c to the minimiser over its captured keys.
 */
uq_status uq_calibrate_c(const void* x, int32_t in_dtype, int64_t n_vec, int32_t head_dim, uint64_t rot_seed,
                         const float* c_list, int32_t n_c, int32_t mode, double* sse, cudaStream_t stream);

/*
 * Cascade (shared-prefix) decode over an FP4 cache.  Agent sessions reuse one
 * long prefix across many sequences and turns ([UQ-review] §1); sequences that
 * reference the same prefix pages can read and convert them once for all.
 * The result equals uq_decode_attention on the same arguments (up to the
 * order of fp32 additions) whenever the promise below holds.
 * cu_seqs     : device int32 [num_groups + 1], non-decreasing, cu_seqs[0] = 0,
 *               cu_seqs[num_groups] <= batch: group g is sequences
 *               cu_seqs[g] .. cu_seqs[g+1]-1; later sequences belong to no group.
 * prefix_lens : device int32 [num_groups].  PROMISE: keys 0 .. prefix_lens[g]-1
 *               of every sequence of group g sit on the same pages (the block
 *               table rows agree there).  The pages are read from the row of the
 *               group's first sequence.  prefix_lens[g] <= seq_lens[b] for each b
 *               of the group (a violation is recorded as UQ_ERR_DEVICE_BOUNDS).
 * max_prefix_len : host bound on prefix_lens (sizes the work split; larger
 *               prefixes are cut to it, the rest going to the per-sequence part).
 * min_rows    : a group is attended once only if it has at least min_rows
 *               query rows (sequences x num_q_heads / num_kv_heads); smaller
 *               groups run as a plain decode.  The shared-prefix kernel
 *               (tensor-core tiles of 128 query rows) is faster than the decode
 *               from about 128 rows (measured at 98304 shared of 131072 keys:
 *               0.91x the plain decode's speed at 64 rows, 1.45x at 128).
 * Work split: group g's first S_g = floor(min(prefix_lens[g], max_prefix_len,
 * max_pages_per_seq * page_size) / 16) * 16 keys go to the shared-prefix kernel
 * (all the group's queries at once); keys S_g .. seq_lens[b]-1 of each sequence
 * to the decode; a log-sum-exp merge combines both, then rotates back.
 * Other arguments as uq_decode_attention; workspace at least
 * uq_cascade_workspace_bytes(batch, num_groups, num_q_heads, num_kv_heads,
 * head_dim, max_prefix_len).  FP4 caches, head_dim 64 or 128.
 */
size_t uq_cascade_workspace_bytes(int32_t batch, int32_t num_groups, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t max_prefix_len);
uq_status uq_cascade_decode_attention(const void* q, const uq_cache* cache, const int32_t* block_table,
                                      int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                                      int32_t num_q_heads, const int32_t* cu_seqs, const int32_t* prefix_lens,
                                      int32_t num_groups, int32_t max_prefix_len, int32_t min_rows,
                                      float sm_scale, float* out, void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream);

/*
 * The TQ4 codebook ([TQ-guide] "랜덤 회전과 Beta 분포", "Lloyd-Max 스칼라 양자화
 * (Q_mse)"): the Lloyd-Max quantiser with 2^bits levels of one coordinate of
 * a uniformly random unit vector in R^head_dim, whose density is
 * Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)) (1 - x^2)^((d-3)/2).  Computed on the
 * host in double precision (the two optimality conditions alternated on the
 * half-line until no centroid moves by 1e-14 standard deviations), symmetric.
 * magnitudes : host float [2^(bits-1)], the non-negative centroids ascending,
 *              each rounded to the nearest f16 (the values the cache decodes to).
 * thresholds : host float [2^bits - 1], the fp32 roundings of the midpoints
 *              between consecutive centroids, ascending (the middle one is 0).
 * bits in 1..4, head_dim in 16..1024.  Host-only; enqueues nothing.  The TQ4
 * cache uses bits = 4 with the cache's head_dim.
 */
uq_status uq_tq_codebook(int32_t head_dim, int32_t bits, float* magnitudes, float* thresholds);

/* The same decode attention for callers that cannot allocate device memory
 * (no counterpart on the pages; a deployment convenience of this library).
 * Some callers cannot provide the workspace: their device memory belongs to
 * another allocator (a framework's caching allocator or a fixed arena) that
 * they may not draw from here, and they may not call cudaMalloc either.  This
 * entry point takes no workspace and allocates nothing: it uses an 8 MiB
 * scratch array compiled into the library, which every GPU that loads the
 * library holds until the process exits.
 *   - Arguments, results and errors are those of uq_decode_attention.
 *   - Batch shapes whose smallest workspace exceeds 8 MiB (roughly more than
 *     2000 (sequence, kv head) pairs at head_dim 128) return UQ_ERR_WORKSPACE
 *     before anything is enqueued; use uq_decode_attention for those.
 *   - batch > 4096 returns UQ_ERR_UNSUPPORTED, as uq_decode_attention does.
 *   - The first call on a device looks up the scratch array's device address
 *     (with that device current), and so does the first call after the
 *     device's context was replaced (cudaDeviceReset); make such a call before
 *     any stream capture.
 *   - All calls on a device share the one scratch array, and it keeps the last
 *     call's contents.  Nothing in it needs to start at zero: every entry a
 *     call reads was written earlier in the same call.  Calls that overlap on
 *     the GPU (different streams, no ordering between them) race on the
 *     scratch and give wrong results; order them on one stream or with
 *     events. */
uq_status uq_decode_attention_noalloc(const void* q, const uq_cache* cache, const int32_t* block_table,
                                      int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                                      int32_t num_q_heads, float sm_scale, float* out, cudaStream_t stream);

/* Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns UQ_OK, UQ_ERR_DEVICE_TIMEOUT or UQ_ERR_DEVICE_BOUNDS (the
 * first error recorded since the last call), or UQ_ERR_CUDA.  After
 * UQ_ERR_DEVICE_TIMEOUT the outputs of the calls since the previous check are
 * undefined (a block that gave up left its part of the result unwritten);
 * after UQ_ERR_DEVICE_BOUNDS the offending accesses were skipped or clamped as
 * each entry point describes. */
uq_status uq_check_device_status(cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* uq_status_string(uq_status status);

/* The ±1 sign diagonal of the rotation, written to host_out[0..d): sign i is
 * -1 when bit 63 of output i of splitmix64 seeded with `seed` is set
 * (Steele, Lea, Flood 2014).  Host-only. */
void uq_rotation_signs(uint64_t seed, int32_t d, int8_t* host_out);

/* ---- test hooks: single stages of the path, for bit-exact checks ---------
 * All pointers are device pointers; d is 64, 128 or 256. */

/* Rotation of n_vec fp32 rows ([UQ-review] §3.1; [TQ-guide] randomised
 * Hadamard rotation and its orthogonality).  x, y: device fp32 [n_vec][d].
 *   inverse = 0: the append's forward rotation, y = fl32(FWHT(s .* x) * fl32(1/sqrt d)).
 *   inverse = 1: the decode's output stage, y = s .* fl32(FWHT(x) * fl32(1/sqrt d))
 *                (the same device code as the merge kernels run).
 * Any other inverse value: UQ_ERR_INVALID_ARG. */
uq_status uq_test_rotate(const float* x, int64_t n_vec, int32_t d, uint64_t seed, int32_t inverse, float* y,
                         cudaStream_t stream);

/* Quantiser stage alone on already-rotated fp32 rows: codes [n_vec][d/2],
 * scales [n_vec][d/32] exactly as in uq_quantize_append. */
uq_status uq_test_quantize_rotated(const float* y, int64_t n_vec, int32_t d, uint8_t* codes,
                                   uint8_t* scales, cudaStream_t stream);

/* The decode prologue alone: rotated, E4M3-rounded query bytes [n_vec][d]
 * from bf16 rows q [n_vec][d]. */
uq_status uq_test_query_fp8(const void* q, int64_t n_vec, int32_t d, uint64_t seed, uint8_t* out,
                            cudaStream_t stream);

/* E4M3 round-to-nearest-even, saturating, of n fp32 values (n even). */
uq_status uq_test_cvt_e4m3(const float* x, int64_t n, uint8_t* out, cudaStream_t stream);

/* The append's E2M1 conversion alone ([UQ-review] §3.1: values rounded to the
 * nearest FP4 E2M1 grid point): codes[i] = code of r[i] (device fp32 [n], n
 * even), round to nearest with ties to the even code, saturating at +-6;
 * bits 0..2 the magnitude rank of {0, .5, 1, 1.5, 2, 3, 4, 6}, bit 3 the IEEE
 * sign bit of r[i].  This is the conversion the append applies to y * 2^-E. */
uq_status uq_test_cvt_e2m1(const float* r, int64_t n, uint8_t* codes, cudaStream_t stream);

/* The append's UE8M0 scale byte alone ([UQ-review] §3.1/§3.3): bytes[i] = the
 * byte of a 32-channel group whose absolute maximum is |m[i]| (device fp32
 * [n]): E = integer nearest to log2(fl32(0.156f * |m|)), byte = clamp(E + 127,
 * 0, 254); 0 for m = 0; 0xFF for a NaN or infinite m. */
uq_status uq_test_scale_byte(const float* m, int64_t n, uint8_t* bytes, cudaStream_t stream);

/* Injected decode timeout: the device-side failure path, exercised without a
 * GPU fault.  Arms the next decode launch that runs the warp-level decode
 * kernel (uq_decode_attention, _append, _noalloc and the cascade's decode, any
 * cache dtype; not the opt-in tensor-memory FP4 decode, which ignores it):
 * warp 0 of block `cta` also waits, at its first unit, on a shared-memory
 * barrier that nothing arrives at, for at most budget_cycles SM clock cycles
 * (plus at most one hardware suspend interval of the wait instruction).  The
 * wait runs out; the kernel records UQ_ERR_DEVICE_TIMEOUT in the device status
 * word, waits (bounded) for that warp's copies in flight and ends the block's
 * work.  That call's output is undefined and the next uq_check_device_status
 * returns UQ_ERR_DEVICE_TIMEOUT; later calls are unaffected (one launch only).
 * If block `cta` or its warp 0 has no units, nothing happens.  Host-only:
 * returns UQ_ERR_INVALID_ARG for cta < 0 or budget_cycles < 0, else UQ_OK. */
uq_status uq_test_arm_decode_timeout(int32_t cta, int64_t budget_cycles);

#ifdef __cplusplus
}
#endif

#endif /* UQ_H_ */
