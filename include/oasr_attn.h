/*
 * oasr_attn.h - C ABI of the paged-KV chunk attention library for GB300 (sm_103a).
 *
 * One hot path of a streaming ASR encoder (OASR documentation pages):
 *
 *   - ASR Engine page, section 4.3 "Batched paged forward": a lockstep cohort of B
 *     streams shares one stacked block_table (B, blocks_per_seq) and one
 *     cache_seqlens (B,) across every layer's paged K/V cache; each step writes the
 *     new chunk into the pool through the block table and the caller commits the
 *     cache length afterwards.
 *   - Scheduler page, section 4.3 "Heterogeneous-offset batching": the attention
 *     over the paged pool masks each stream by its cache_seqlens and adds the
 *     Transformer-XL position term matrix_bd / sqrt(d_k) to the content score.
 *   - Model Layer page, table "Three optional encoder declarations", row
 *     fixed_attention_window: with a uniform cache length one relative-position
 *     table serves the whole cohort, its distances being cache + i - j.
 *   - Model Layer page, Nemotron ASR section: Transformer-XL relative position with
 *     rel_shift.
 *   - ASR Engine page, section 4.1: with sequence packing an offline micro-batch is
 *     one gapless varlen-attention row.
 *
 * Layouts (row-major, innermost last; every pointer is DEVICE memory owned by the
 * caller; the library keeps no pointer after a call returns):
 *   q, k_new, v_new, out (streaming) : [B, T, H, D]
 *   k_pool, v_pool                   : [num_blocks, block_size, H, D]
 *   block_table                      : int32 [B, max_blocks_per_seq]
 *   cache_seqlens                    : int32 [B]  (frames cached BEFORE this chunk)
 *   pos_bias_u, pos_bias_v           : [H, D]
 *   rel                              : [R, H, D]
 *   q, k, v, out (packed)            : [total, H, D]
 *   cu_seqlens                       : int32 [num_seqs + 1], cu[0] = 0, non-decreasing,
 *                                      cu[num_seqs] = total
 * All float tensors of one call share the dtype `dt`.  Base pointers must be 16-byte
 * aligned (the tensor-core path reads them with TMA).
 *
 * The score of query i against key j, for one head, is
 *     s_ij = scale * ( (q_i + u) . k_j + (q_i + v) . rel[rho] )
 * followed by a softmax over j and a weighted sum of the value rows.  The rel row is
 * rho = z - dist in rel_shift order (row 0 holds the largest distance):
 *     streaming: dist = C + i - j, z = R - T, keys j in [0, C + T) (the whole cache
 *                and the whole chunk; no mask inside the chunk), R >= C + 2T - 1;
 *     packed:    dist = i - j within one segment, z = (R - 1) / 2, R >= 2 Lmax - 1.
 *
 * Execution: every call is asynchronous and stream-ordered on `stream`; none
 * synchronises, none allocates device memory.  Host-side argument checks return
 * OASR_ERR_INVALID_ARG / OASR_ERR_UNSUPPORTED before anything is enqueued.  Device
 * data (block ids, cache_seqlens, cu_seqlens) is not read on the host: an entry that
 * points outside its table makes the kernel skip or clamp that access and set a bit of
 * the device status word (oasr_device_status), never read or write out of bounds.
 */
#ifndef OASR_ATTN_H
#define OASR_ATTN_H

#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    OASR_OK = 0,
    OASR_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, misaligned pointer   */
    OASR_ERR_UNSUPPORTED = 2, /* a size or dtype this build has no kernel for         */
    OASR_ERR_CUDA = 3,        /* a CUDA runtime call or a kernel launch failed         */
    OASR_ERR_BOUNDS = 4,      /* (oasr_device_status) a device index was out of range  */
    OASR_ERR_TIMEOUT = 5      /* (oasr_device_status) a kernel wait ran out of time    */
} oasr_status;

typedef enum { OASR_F32 = 0, OASR_BF16 = 1 } oasr_dtype;

/*
 * Paged append (ASR Engine page, section 4.3, step 1: the chunk's rows go into each
 * stream's pool blocks through its block_table).
 *
 * For b < B, t < T, h < H: logical position p = cache_seqlens[b] + t is written to
 * block block_table[b][p / block_size], slot p % block_size:
 *     k_pool[blk][slot][h][:] = k_new[b][t][h][:],  v_pool likewise.
 * A pure copy (bit-exact).  cache_seqlens is read, never advanced: the caller commits
 * the chunk afterwards.  Rows whose position lies past max_blocks_per_seq pages, or whose
 * block id is outside [0, num_blocks), are skipped (status bit OASR_ERR_BOUNDS).
 * D * sizeof(dtype) must be a multiple of 16 bytes and 2 * B * T at most 2^26 (else
 * OASR_ERR_UNSUPPORTED).
 */
oasr_status oasr_paged_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                              int num_blocks, int block_size, const int32_t* block_table,
                              int max_blocks_per_seq, const int32_t* cache_seqlens, int B,
                              int T, int H, int D, oasr_dtype dt, cudaStream_t stream);

/*
 * Streaming chunk attention over the paged pool (Scheduler page, section 4.3; Model
 * Layer page, fixed_attention_window row; Nemotron ASR section).
 *
 * For every stream b, head h and chunk row i < T, attends over the C_b + T keys that
 * the pool holds for stream b (C_b = cache_seqlens[b]: the cached frames followed by
 * this chunk, which oasr_paged_append must already have written on the same stream)
 * and writes out[b][i][h][:].  Requirements: D = 64; 1 <= T <= 64; block_size a power of
 * two in [8, 256]; R >= max_b C_b + 2T - 1; C_b + T <= max_blocks_per_seq * block_size.
 * A stream that breaks either raises the status bit OASR_ERR_BOUNDS and its row is then
 * unspecified: the bf16 path drops its keys past min(max_blocks_per_seq * block_size,
 * R - T + 1) (the keys the host can bound, for which it sizes its shared memory, so an
 * engine-sized block table costs nothing), the f32 path drops keys past the table's pages
 * and reads zero rows for the distances the rel table lacks.  scale is normally 1/sqrt(D).
 * bf16: bf16 inputs, fp32 accumulation and softmax, bf16 output rounded once; chunks of
 * 33 to 64 frames with an even H run on the 5th-generation tensor cores (two heads of a
 * stream per 128-row tile), other shapes on the legacy mma.sync path.
 * f32: fp32 throughout (no TF32).
 */
oasr_status oasr_chunk_relattn_paged(const void* q, const void* k_pool, const void* v_pool,
                                     int num_blocks, int block_size,
                                     const int32_t* block_table, int max_blocks_per_seq,
                                     const int32_t* cache_seqlens, const void* pos_bias_u,
                                     const void* pos_bias_v, const void* rel, int R, void* out,
                                     int B, int T, int H, int D, float scale, oasr_dtype dt,
                                     cudaStream_t stream);

/*
 * One fused streaming step: oasr_paged_append followed by oasr_chunk_relattn_paged, in
 * one launch.  Each (stream, head) program writes its head's slice of the chunk into
 * the pool and then attends over cache + chunk, so the chunk is never re-read from
 * HBM (when every page the chunk lands in is a valid block, the attention reads the
 * chunk's keys straight from k_new / v_new).  For bf16 chunks of 33 to 64 frames with an
 * even H the step is instead the two calls in sequence on `stream` (the append, then the
 * tensor-core attention over the pool).  Results equal the two calls in sequence up to
 * floating-point summation order; the pool afterwards is bit-identical.  The same
 * requirements apply.  Block ids of different streams must not alias a block that this
 * step writes.
 */
oasr_status oasr_chunk_step_paged(const void* q, const void* k_new, const void* v_new,
                                  void* k_pool, void* v_pool, int num_blocks, int block_size,
                                  const int32_t* block_table, int max_blocks_per_seq,
                                  const int32_t* cache_seqlens, const void* pos_bias_u,
                                  const void* pos_bias_v, const void* rel, int R, void* out,
                                  int B, int T, int H, int D, float scale, oasr_dtype dt,
                                  cudaStream_t stream);

/*
 * Packed varlen bidirectional attention (ASR Engine page, section 4.1; Model Layer
 * page, engine-facing surface table, forward_offline_packed).
 *
 * Segment s owns rows [cu_seqlens[s], cu_seqlens[s+1]); each of its queries attends to
 * every key of the same segment, with distance i - j (local indices) and rel row
 * z - (i - j), z = (R - 1) / 2.  Requirements: D = 64; 1 <= num_seqs <= 1024;
 * max_seqlen >= every segment length; R >= 2 * max_seqlen - 1; bf16: (total / 128 +
 * num_seqs) * H < 2^31 (else OASR_ERR_UNSUPPORTED).  Rows of a segment that would cross
 * `total` are clamped (status bit OASR_ERR_BOUNDS).
 */
oasr_status oasr_packed_relattn_varlen(const void* q, const void* k, const void* v,
                                       const int32_t* cu_seqlens, int num_seqs, int max_seqlen,
                                       int total, const void* pos_bias_u,
                                       const void* pos_bias_v, const void* rel, int R, void* out,
                                       int H, int D, float scale, oasr_dtype dt,
                                       cudaStream_t stream);

/*
 * Chunked-limited packed attention: the Nemotron offline mask (Model Layer page, Nemotron
 * ASR section: the chunked_limited mask applies offline too; a query sees its own chunk of
 * num_lookahead_tokens + 1 frames plus (sliding_window - 1) // chunk earlier chunks, and
 * the offline pass scores each query block against its own frames plus that history).
 *
 * As oasr_packed_relattn_varlen, but query i of a segment attends to key j only when
 * i / chunk_size - left_chunks <= j / chunk_size <= i / chunk_size (positions local to the
 * segment, integer division): chunk_size = num_lookahead_tokens + 1, left_chunks =
 * (sliding_window - 1) / chunk_size.  The work done grows with the segment length, not its
 * square.  Requirements as for oasr_packed_relattn_varlen, plus chunk_size >= 1 and
 * left_chunks >= 0 (else OASR_ERR_INVALID_ARG).  A chunk_size of at least every segment
 * length gives the bidirectional attention, up to summation order: in bf16 with an even head
 * count and at most 511 segments the call runs a tensor-core kernel of its own (64 queries
 * of a segment for a pair of heads per tile), otherwise the one-head packed kernel.
 */
oasr_status oasr_packed_relattn_chunked(const void* q, const void* k, const void* v,
                                        const int32_t* cu_seqlens, int num_seqs, int max_seqlen,
                                        int total, const void* pos_bias_u,
                                        const void* pos_bias_v, const void* rel, int R, void* out,
                                        int H, int D, float scale, int chunk_size,
                                        int left_chunks, oasr_dtype dt, cudaStream_t stream);

/*
 * Commit a streaming step with fixed-window history eviction (ASR Engine page, KV-pool sizing
 * paragraphs: an encoder with a trained attention window pages by chunk and retains
 * ceil(window / chunk) + 1 pages per stream; with eviction the cached length is held at the
 * window; section 4.3: the caller commits the cache length after the step).
 *
 * For every stream b, after a chunk of T frames was appended at cache_seqlens[b], the stream
 * holds n = cache_seqlens[b] + T frames in its first P = ceil(n / block_size) pages.  If
 * n > window_frames, the oldest d = min(ceil((n - window_frames) / block_size),
 * floor(n / block_size)) pages are dropped (whole pages only: a partly written newest page
 * stays, so with a window shorter than a page the cached length may exceed the window by
 * less than a page and is never negative): block_table[b][0 .. P) is rotated left by d, so
 * the dropped blocks become the next pages to be written, and cache_seqlens[b] becomes
 * n - d * block_size; otherwise cache_seqlens[b] becomes n.  Entries past the first P are
 * untouched.  Both arrays are device memory and are
 * updated in place on `stream`, so a captured step stays replayable.
 *
 * Requirements: B >= 1; 1 <= max_blocks_per_seq <= 512 (else OASR_ERR_UNSUPPORTED);
 * block_size >= 1; T >= 0; window_frames >= 0.  A negative cache length or a row that would
 * run past the table raises OASR_ERR_BOUNDS in the device status word and is clamped.
 */
oasr_status oasr_window_commit(int32_t* block_table, int32_t* cache_seqlens, int B,
                               int max_blocks_per_seq, int block_size, int T, int window_frames,
                               cudaStream_t stream);

/*
 * The projections that feed the path, in one launch (Model Layer page, fixed_attention_window
 * row: one positional projection per step serves the cohort; the Conformer rel-pos attention's
 * linear_q / linear_k / linear_v carry a bias, linear_pos does not):
 *
 *   q | k | v = x . w_qkv^T + b_qkv     x [M, d_model], w_qkv [3 d_model, d_model] (q rows,
 *                                       then k, then v), b_qkv [3 d_model]; q, k, v written as
 *                                       [M, H, 64] (M = B * T frames: the [B, T, H, 64] inputs of
 *                                       the attention calls)
 *   rel       = pos_emb . w_pos^T        pos_emb [R, d_model], w_pos [d_model, d_model]; rel
 *                                       written as [R, H, 64]
 *
 * bf16 in and out, fp32 accumulation, one rounding per output.  Requirements: d_model = 64 H
 * and a multiple of 128 (else OASR_ERR_UNSUPPORTED); every pointer 16-byte aligned.
 */
oasr_status oasr_project_qkv_pos(const void* x, const void* w_qkv, const void* b_qkv,
                                 const void* pos_emb, const void* w_pos, void* q, void* k, void* v,
                                 void* rel, int M, int R, int d_model, int H, oasr_dtype dt,
                                 cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* oasr_status_string(oasr_status status);

/*
 * Device status word of the current device: an OR of OASR_ERR_BOUNDS (bit 0) and
 * OASR_ERR_TIMEOUT (bit 1) flags raised by kernels since the last clear.  Synchronises
 * the current device first.  *flags receives the raw bits (1 = bounds, 2 = timeout); if
 * clear is non-zero the word is reset to 0.  Returns OASR_ERR_CUDA if the read fails.
 */
oasr_status oasr_device_status(unsigned* flags, int clear);

/*
 * Diagnostic (the pages have no counterpart): run the library's bounded pipeline wait on a
 * barrier that nothing ever signals, with a limit of limit_us microseconds (1 .. 2000000),
 * on `stream`.  One CTA of one warp; when the wait runs out it raises the timeout bit of the
 * device status word and returns, as a kernel of the library does when a copy it waits for
 * never lands.  The context stays usable.  Returns OASR_ERR_INVALID_ARG for a limit outside
 * the range (nothing is launched), OASR_ERR_CUDA if the launch fails.
 */
oasr_status oasr_selftest_wait(unsigned limit_us, cudaStream_t stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int oasr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OASR_ATTN_H */
