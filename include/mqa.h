/*
 * mqa.h -- C ABI of libmqa.so: the incremental decode step of Multi-Query / Grouped-Query
 * Attention on NVIDIA B300 (sm_103a).
 *
 * Notation (from "分组查询注意力（GQA）与多查询注意力（MQA）深度实战", ybb.press, §四/§五):
 *   b     sequences in the batch
 *   h     query heads;  g = num_kv_heads  (g = h is MHA, g = 1 is MQA), h % g == 0
 *   G     = h / g, the query heads that share one K/V head; query head i reads KV head
 *           j = i / G, so the heads of one group are contiguous
 *   d_h   head dimension (64 or 128)
 *   n_max rows allocated per (sequence, KV head) in the cache
 *
 * Memory layout (all row-major, no padding, every tensor on the current CUDA device):
 *   q, out           [b][h][d_h]            bfloat16
 *   k_new, v_new     [b][g][d_h]            bfloat16
 *   k_cache, v_cache [b][g][n_max][d_h]     bfloat16
 *   pos, seq_lens    [b]                    int32
 * bfloat16 values travel as their 16-bit patterns (mqa_bf16).
 *
 * Ownership: the caller allocates and owns every buffer; the library keeps no pointer to them
 * after a call returns. The library owns one internal workspace per (device, stream) for the
 * split-sequence partial results of mqa_decode_attention; it grows on demand (cudaMalloc, so
 * the first call at a new, larger shape must happen outside CUDA-graph capture) and lives until
 * the process exits.
 *
 * Ordering and errors: both compute calls only enqueue work on `stream` (a cudaStream_t; NULL
 * is the legacy default stream) and return before the GPU has finished. Call mqa_kv_append
 * before mqa_decode_attention on the same stream so that attention sees the new row. Arguments
 * are checked on the host before anything is enqueued; a failed check returns an error code and
 * enqueues nothing. Problems only the GPU can see (a position or length out of range, an
 * internal wait that timed out) are latched in a per-device status word that
 * mqa_get_device_status() reads; such a sequence's output is written as zeros and its cache is
 * left untouched -- nothing is truncated silently. No C++ exception crosses this boundary.
 */
#ifndef MQA_H_
#define MQA_H_

#include <stdint.h>

#if defined(__GNUC__)
#define MQA_API __attribute__((visibility("default")))
#else
#define MQA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mqa_bf16;

typedef enum mqa_status {
  MQA_OK = 0,
  MQA_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, non-positive size, h % g != 0, ... */
  MQA_ERR_UNSUPPORTED = 2,    /* a valid request outside what the kernels implement */
  MQA_ERR_CUDA = 3,           /* a CUDA runtime call or kernel launch failed */
  MQA_ERR_DEVICE_BOUNDS = 4,  /* (latched) a pos, seq_lens or used page-table entry was out of range */
  MQA_ERR_TIMEOUT = 5         /* (latched) an in-kernel wait exceeded its time limit */
} mqa_status;

/*
 * mqa_kv_append -- write this step's K and V rows into the cache.
 *
 * Defined by the decode step of "GQA与MQA深度实战" (ybb.press) §八, which stores the new token's
 * K/V for the g KV heads at the current position before attending, and by the
 * nanhubrain.csdn.net MQA article §2.2, which concatenates the new row onto the cached K/V
 * along the sequence axis.
 *
 * For every sequence bi < b and KV head j < g:
 *     k_cache[bi][j][pos[bi]][:] = k_new[bi][j][:]      (and the same for V)
 * The copy is bit-exact; every other byte of both caches is left unchanged.
 *
 *   k_new, v_new     device, [b][g][d_h] bf16, 16-byte aligned, read only
 *   k_cache, v_cache device, [b][g][n_max][d_h] bf16, 16-byte aligned, updated in place
 *   pos              device, [b] int32, the row to write, 0 <= pos[bi] < n_max
 *   b, g, d_h, n_max sizes (> 0; d_h in {64, 128})
 *   stream           cudaStream_t to enqueue on
 *
 * Returns MQA_OK, MQA_ERR_INVALID_ARG, MQA_ERR_UNSUPPORTED or MQA_ERR_CUDA. A pos entry outside
 * [0, n_max) skips that sequence and latches MQA_ERR_DEVICE_BOUNDS.
 */
MQA_API int mqa_kv_append(const mqa_bf16* k_new, const mqa_bf16* v_new, mqa_bf16* k_cache,
                  mqa_bf16* v_cache, const int32_t* pos, int b, int g, int d_h, int n_max,
                  void* stream);

/*
 * mqa_decode_attention -- grouped scaled-dot-product attention of one new query token per
 * sequence against its cached keys and values.
 *
 * Defined by "GQA与MQA深度实战" (ybb.press) §五: with j = i / (h/g),
 *     score_{i,t} = scale * q_i . K_{j,t},   alpha_{i,t} = softmax_t(score_{i,t}),
 *     O_i = sum_t alpha_{i,t} V_{j,t};
 * the page's scale is 1/sqrt(d_h). The sum runs over the rows t < seq_lens[bi] of sequence bi,
 * which include the row appended this step (the page's §八 module attends over every cached
 * position up to and including the new one). Rows at or beyond seq_lens[bi] are never read into
 * the result, whatever they hold.
 *
 * Inputs are bf16, products and sums are fp32, `out` is rounded to bf16 (nearest-even). The
 * result matches the fp64 definition within the tolerances stated by the tests.
 *
 *   q                device, [b][h][d_h] bf16, 16-byte aligned, read only
 *   k_cache, v_cache device, [b][g][n_max][d_h] bf16, 16-byte aligned, read only
 *   seq_lens         device, [b] int32, 1 <= seq_lens[bi] <= n_max
 *   out              device, [b][h][d_h] bf16, 16-byte aligned, written
 *   b, h, g          sizes (> 0, h % g == 0, h / g <= 64, b <= 8192)
 *   d_h              64 or 128
 *   n_max            cache rows per (sequence, KV head), > 0
 *   scale            finite logit scale (normally 1/sqrt(d_h))
 *   stream           cudaStream_t to enqueue on
 *
 * Returns MQA_OK, MQA_ERR_INVALID_ARG, MQA_ERR_UNSUPPORTED or MQA_ERR_CUDA. A seq_lens entry
 * outside [1, n_max] writes zeros for that sequence and latches MQA_ERR_DEVICE_BOUNDS. Two calls
 * that share a stream share that stream's workspace and are ordered by the stream; calls on
 * different streams use different workspaces.
 */
MQA_API int mqa_decode_attention(const mqa_bf16* q, const mqa_bf16* k_cache, const mqa_bf16* v_cache,
                         const int32_t* seq_lens, mqa_bf16* out, int b, int h, int g, int d_h,
                         int n_max, float scale, void* stream);

/*
 * mqa_decode_step -- one whole decode step of one layer in a single launch: the append of
 * mqa_kv_append followed by the attention of mqa_decode_attention, with the same result as
 * calling the two in that order on one stream (the cache rows bit for bit, `out` within the
 * same tolerances).
 *
 * Defined by the decode step of "GQA与MQA深度实战" (ybb.press) §八 (store the new token's K/V at
 * the current position, then attend over every cached row up to and including it) and §五 (the
 * grouped attention, see mqa_decode_attention); the nanhubrain.csdn.net MQA article §2.2 orders
 * the append before the attention in the same way.
 *
 * The new rows are written by the CTA that loads the tile holding them, immediately before that
 * tile is copied into shared memory, so the step reads each cache row once and launches once.
 *
 *   q, out           as for mqa_decode_attention
 *   k_new, v_new     device, [b][g][d_h] bf16, 16-byte aligned, read only
 *   k_cache, v_cache device, [b][g][n_max][d_h] bf16, 16-byte aligned; row pos[bi] of every
 *                    (bi, j) is written, every other row only read
 *   pos              device, [b] int32, 0 <= pos[bi] < n_max
 *   seq_lens         device, [b] int32, 1 <= seq_lens[bi] <= n_max; normally pos[bi] + 1
 *   b, h, g, d_h, n_max, scale, stream   as for mqa_decode_attention
 *
 * Returns MQA_OK, MQA_ERR_INVALID_ARG, MQA_ERR_UNSUPPORTED or MQA_ERR_CUDA. A pos entry out of
 * range skips that sequence's append; a seq_lens entry out of range writes zeros for that
 * sequence's output; both latch MQA_ERR_DEVICE_BOUNDS. The workspace is that of
 * mqa_decode_attention (shared per stream).
 */
MQA_API int mqa_decode_step(const mqa_bf16* q, const mqa_bf16* k_new, const mqa_bf16* v_new,
                            mqa_bf16* k_cache, mqa_bf16* v_cache, const int32_t* pos,
                            const int32_t* seq_lens, mqa_bf16* out, int b, int h, int g, int d_h,
                            int n_max, float scale, void* stream);

/*
 * Paged caches: mqa_kv_append_paged, mqa_decode_attention_paged, mqa_decode_step_paged.
 *
 * The same three operations over a cache kept in fixed-size pages found through a per-sequence
 * page table, the layout serving stacks use for ragged batches: the nanhubrain.csdn.net MQA
 * article §3.3 describes vLLM's PagedAttention cutting the cache into pages of 16 tokens by
 * default, and "GQA与MQA深度实战" (ybb.press) §十 item 12 pairs ragged per-request lengths with
 * such paging. The pages fix no layout; this library's reading:
 *
 *   k_pool, v_pool   device, [num_pages][g][page_size][d_h] bf16, 16-byte aligned: page p holds
 *                    page_size consecutive rows of every KV head
 *   page_table       device, [b][max_pages] int32: row t of sequence bi (every KV head j) is row
 *                    t % page_size of page page_table[bi][t / page_size], i.e.
 *                    K[bi][j][t] = k_pool[page_table[bi][t / page_size]][j][t % page_size]
 *   page_size        a power of two, at least 8 (else MQA_ERR_UNSUPPORTED)
 *   max_pages        entries per table row; a sequence addresses n_max = max_pages * page_size
 *                    rows (max_pages * page_size <= 2^31 - 1)
 *   num_pages        pages in each pool (num_pages * g < 2^31 - 1)
 *
 * Each call computes exactly what its contiguous counterpart computes on the cache the table
 * describes (the rows above, gathered into [b][g][n_max][d_h]); the tests compare the two through
 * the oracle's gather. Only the table entries of pages a call touches are used: those holding
 * rows t < seq_lens[bi] (attention) and row pos[bi] (append), so entries past a sequence's last
 * page may hold anything (-1 for "no page", say; the table is read a batch of tiles ahead, so such
 * entries may be loaded, but their values never matter). A used entry outside [0, num_pages) latches
 * MQA_ERR_DEVICE_BOUNDS; its rows read as zeros in attention and its append is skipped. Pages
 * may be shared between sequences (a common prefix) and read by all of them, but a page that a
 * call appends to must not be read by another sequence in the same call, and two sequences must
 * not append to the same row: the order of those accesses is not defined. Only the mma.sync and
 * CUDA-core paths read paged caches: with mqa_debug_override forcing path 3 (tcgen05) the paged
 * attention and step calls return MQA_ERR_UNSUPPORTED. Everything else -- argument meaning,
 * ownership, ordering, the workspace, the status word -- is as for the contiguous calls.
 */
MQA_API int mqa_kv_append_paged(const mqa_bf16* k_new, const mqa_bf16* v_new, mqa_bf16* k_pool,
                                mqa_bf16* v_pool, const int32_t* pos, const int32_t* page_table,
                                int b, int g, int d_h, int page_size, int max_pages,
                                int num_pages, void* stream);
MQA_API int mqa_decode_attention_paged(const mqa_bf16* q, const mqa_bf16* k_pool,
                                       const mqa_bf16* v_pool, const int32_t* page_table,
                                       const int32_t* seq_lens, mqa_bf16* out, int b, int h,
                                       int g, int d_h, int page_size, int max_pages,
                                       int num_pages, float scale, void* stream);
MQA_API int mqa_decode_step_paged(const mqa_bf16* q, const mqa_bf16* k_new,
                                  const mqa_bf16* v_new, mqa_bf16* k_pool, mqa_bf16* v_pool,
                                  const int32_t* pos, const int32_t* page_table,
                                  const int32_t* seq_lens, mqa_bf16* out, int b, int h, int g,
                                  int d_h, int page_size, int max_pages, int num_pages,
                                  float scale, void* stream);

/*
 * fp8 caches: mqa_kv_append_fp8, mqa_decode_attention_fp8, mqa_decode_step_fp8.
 *
 * The same three operations over caches that hold 8-bit floating-point codes (E4M3: 1 sign, 4
 * exponent and 3 fraction bits, exponent bias 7, no infinities, largest finite value 448) with
 * one scale per tensor: an element's value is code * k_scale (K) or code * v_scale (V). This
 * halves the bytes the bandwidth-bound path reads. The pages discuss quantizing the K/V cache
 * ("GQA与MQA深度实战" (ybb.press) §十 item 7; the nanhubrain.csdn.net MQA article §4.3 warns that
 * K/V shared by many query heads makes quantization error count more) but fix no format; this
 * library's reading is E4M3 with per-tensor scales, the scales chosen by the caller.
 *
 *   k_cache, v_cache device, [b][g][n_max][d_h] uint8 E4M3 codes, 16-byte aligned
 *   k_scale, v_scale finite and > 0 (else MQA_ERR_INVALID_ARG)
 *   d_h              128 (else MQA_ERR_UNSUPPORTED)
 *   everything else  as for the bf16 calls
 *
 * Append: for every element x of k_new[bi][j] (bf16), the code written is
 * E4M3(fp32(x) / k_scale), the division rounded once in fp32 and the result rounded to the nearest
 * E4M3 value, ties to even, magnitudes beyond 448 saturating to +-448 (V likewise with v_scale).
 * Attention: as mqa_decode_attention over the values code * scale. q stays bf16 (rounded to fp16
 * for the tensor-core products), the codes are widened exactly, products and sums are fp32, and
 * the result matches the fp64 attention over the dequantized caches within the tolerances the
 * tests state. The tcgen05 path does not read fp8 caches (path 3 returns MQA_ERR_UNSUPPORTED).
 */
MQA_API int mqa_kv_append_fp8(const mqa_bf16* k_new, const mqa_bf16* v_new, uint8_t* k_cache,
                              uint8_t* v_cache, const int32_t* pos, int b, int g, int d_h,
                              int n_max, float k_scale, float v_scale, void* stream);
MQA_API int mqa_decode_attention_fp8(const mqa_bf16* q, const uint8_t* k_cache,
                                     const uint8_t* v_cache, const int32_t* seq_lens,
                                     mqa_bf16* out, int b, int h, int g, int d_h, int n_max,
                                     float scale, float k_scale, float v_scale, void* stream);
MQA_API int mqa_decode_step_fp8(const mqa_bf16* q, const mqa_bf16* k_new, const mqa_bf16* v_new,
                                uint8_t* k_cache, uint8_t* v_cache, const int32_t* pos,
                                const int32_t* seq_lens, mqa_bf16* out, int b, int h, int g,
                                int d_h, int n_max, float scale, float k_scale, float v_scale,
                                void* stream);

/*
 * Several new tokens per sequence: mqa_kv_append_multi, mqa_decode_attention_multi,
 * mqa_decode_step_multi.
 *
 * The decode step for T tokens at once (draft tokens of speculative decoding, or a chunk of a
 * prompt): "GQA与MQA深度实战" (ybb.press) §八's module takes T new tokens, writes their K/V rows at
 * start .. start + T - 1 and attends over the first start + T rows; its checklist §十 item 10 keeps
 * the causal mask per query position when K/V are shared. Reading: token t (0-based) of sequence bi
 * sits at row L - T + t, where L = seq_lens[bi] counts all T new rows, and attends the first
 * L - T + 1 + t rows; T = 1 is mqa_decode_attention. Every K/V byte is read once for all T tokens.
 *
 *   q, out           device, [b][T][h][d_h] bf16 (token-major), 16-byte aligned
 *   k_new, v_new     device, [b][T][g][d_h] bf16, 16-byte aligned
 *   pos              device, [b] int32: token t is written at row pos[bi] + t;
 *                    0 <= pos[bi] and pos[bi] + T <= n_max, else that sequence is not written
 *   seq_lens         device, [b] int32, T <= seq_lens[bi] <= n_max (normally pos[bi] + T), else
 *                    zeros for that sequence
 *   T                tokens per sequence, >= 1, with T * (h / g) <= 2^22
 *   everything else  as for mqa_kv_append / mqa_decode_attention / mqa_decode_step
 *
 * Two kernels serve these calls, by the rows a KV head's attention has, T * (h / g):
 *   - up to 64 (speculative decoding): the mma.sync decode kernel, the rows of a KV head in one
 *     tile of heads, K/V tiles split across CTAs and merged; the step is one launch;
 *   - more (a prefill-sized T: a prompt chunk): the tcgen05 prefill kernel, 128 rows per
 *     tensor-core tile with accumulators in tensor memory, each block of 128 rows finished by one
 *     CTA; the step is two launches, the append and then the attention, since every block of a
 *     sequence reads its new rows. Forcing the tcgen05 path (mqa_debug_override path 3) sends
 *     every T > 1 call there.
 * A forced CUDA-core path returns MQA_ERR_UNSUPPORTED when T > 1, and so does forced mma.sync past
 * 64 rows. Both latched errors are MQA_ERR_DEVICE_BOUNDS. The decode kernel uses the workspace of
 * mqa_decode_attention; the prefill kernel none.
 */
MQA_API int mqa_kv_append_multi(const mqa_bf16* k_new, const mqa_bf16* v_new, mqa_bf16* k_cache,
                                mqa_bf16* v_cache, const int32_t* pos, int b, int T, int g,
                                int d_h, int n_max, void* stream);
MQA_API int mqa_decode_attention_multi(const mqa_bf16* q, const mqa_bf16* k_cache,
                                       const mqa_bf16* v_cache, const int32_t* seq_lens,
                                       mqa_bf16* out, int b, int T, int h, int g, int d_h,
                                       int n_max, float scale, void* stream);
MQA_API int mqa_decode_step_multi(const mqa_bf16* q, const mqa_bf16* k_new,
                                  const mqa_bf16* v_new, mqa_bf16* k_cache, mqa_bf16* v_cache,
                                  const int32_t* pos, const int32_t* seq_lens, mqa_bf16* out,
                                  int b, int T, int h, int g, int d_h, int n_max, float scale,
                                  void* stream);

/*
 * Paged caches with fp8 codes or with several new tokens: mqa_kv_append_paged_fp8,
 * mqa_decode_attention_paged_fp8, mqa_decode_step_paged_fp8 and mqa_kv_append_paged_multi,
 * mqa_decode_attention_paged_multi, mqa_decode_step_paged_multi.
 *
 * A serving stack keeps its cache in pages and also quantizes it, or verifies several draft
 * tokens at once: the nanhubrain.csdn.net MQA article §3.3 (vLLM's paged blocks) with §4.3
 * question 3 (quantized K/V), and "GQA与MQA深度实战" (ybb.press) §十 items 7 and 12. These calls
 * combine the page layout of the paged calls with the element type of the fp8 calls, or with the
 * T tokens of the several-token calls; each is defined as the operation of the non-paged call on
 * the rows the page table maps:
 *   - pools, table, page_size, max_pages, num_pages: as for mqa_kv_append_paged (n_max of a
 *     sequence is max_pages * page_size);
 *   - the fp8 calls: pools [num_pages][g][page_size][d_h] of E4M3 codes (uint8), d_h = 128,
 *     k_scale and v_scale as for mqa_kv_append_fp8; one new token per sequence;
 *   - the several-token calls: q and out [b][T][h][d_h], k_new and v_new [b][T][g][d_h], token t
 *     of sequence bi written at row pos[bi] + t through the table and attending the first
 *     seq_lens[bi] - T + 1 + t rows; T * (h / g) <= 64 (the mma.sync decode kernel; a larger T
 *     returns MQA_ERR_UNSUPPORTED here: the prefill kernel reads contiguous caches).
 * A pos whose rows do not all fit the table skips that sequence's append, a used page index
 * outside [0, num_pages) skips that row (its attention reads zeros there); both latch
 * MQA_ERR_DEVICE_BOUNDS. The fused steps are one launch and use the workspace of
 * mqa_decode_attention. Returns MQA_OK, MQA_ERR_INVALID_ARG, MQA_ERR_UNSUPPORTED or MQA_ERR_CUDA.
 */
MQA_API int mqa_kv_append_paged_fp8(const mqa_bf16* k_new, const mqa_bf16* v_new,
                                    uint8_t* k_pool, uint8_t* v_pool, const int32_t* pos,
                                    const int32_t* page_table, int b, int g, int d_h,
                                    int page_size, int max_pages, int num_pages, float k_scale,
                                    float v_scale, void* stream);
MQA_API int mqa_decode_attention_paged_fp8(const mqa_bf16* q, const uint8_t* k_pool,
                                           const uint8_t* v_pool, const int32_t* page_table,
                                           const int32_t* seq_lens, mqa_bf16* out, int b, int h,
                                           int g, int d_h, int page_size, int max_pages,
                                           int num_pages, float scale, float k_scale,
                                           float v_scale, void* stream);
MQA_API int mqa_decode_step_paged_fp8(const mqa_bf16* q, const mqa_bf16* k_new,
                                      const mqa_bf16* v_new, uint8_t* k_pool, uint8_t* v_pool,
                                      const int32_t* pos, const int32_t* page_table,
                                      const int32_t* seq_lens, mqa_bf16* out, int b, int h, int g,
                                      int d_h, int page_size, int max_pages, int num_pages,
                                      float scale, float k_scale, float v_scale, void* stream);
MQA_API int mqa_kv_append_paged_multi(const mqa_bf16* k_new, const mqa_bf16* v_new,
                                      mqa_bf16* k_pool, mqa_bf16* v_pool, const int32_t* pos,
                                      const int32_t* page_table, int b, int T, int g, int d_h,
                                      int page_size, int max_pages, int num_pages, void* stream);
MQA_API int mqa_decode_attention_paged_multi(const mqa_bf16* q, const mqa_bf16* k_pool,
                                             const mqa_bf16* v_pool, const int32_t* page_table,
                                             const int32_t* seq_lens, mqa_bf16* out, int b, int T,
                                             int h, int g, int d_h, int page_size, int max_pages,
                                             int num_pages, float scale, void* stream);
MQA_API int mqa_decode_step_paged_multi(const mqa_bf16* q, const mqa_bf16* k_new,
                                        const mqa_bf16* v_new, mqa_bf16* k_pool,
                                        mqa_bf16* v_pool, const int32_t* pos,
                                        const int32_t* page_table, const int32_t* seq_lens,
                                        mqa_bf16* out, int b, int T, int h, int g, int d_h,
                                        int page_size, int max_pages, int num_pages, float scale,
                                        void* stream);

/*
 * mqa_decode_attention_noalloc -- mqa_decode_attention for callers that cannot allocate device
 * memory. The source pages have no counterpart to this call; it exists for users of the library.
 *
 * mqa_decode_attention may call cudaMalloc the first time a stream needs a larger workspace. Some
 * callers cannot allow that. One example is a host framework that has already reserved the
 * device's memory for its own pool, where cudaMalloc fails or fragments that pool. Another is a
 * latency-critical loop that cannot take cudaMalloc's implicit device synchronisation. This
 * variant runs the same kernels and computes the same result. It keeps its scratch (the split
 * partial states) in a fixed array of MQA_NOALLOC_SCRATCH_BYTES inside the library's device
 * memory, which every GPU that loads the library holds until the process exits. The call itself
 * allocates nothing: it calls no cudaMalloc, no cudaFree and no allocating library routine.
 *
 * Arguments, layout, ownership, ordering and errors are those of mqa_decode_attention, plus:
 *   - the array holds MQA_NOALLOC_MAX_SEGMENTS arrival counters (one per sequence and KV head)
 *     followed by the split partial states. A problem with more than MQA_NOALLOC_MAX_SEGMENTS
 *     values of b*g, or whose partial states need more than the rest of the array, returns
 *     MQA_ERR_UNSUPPORTED and enqueues nothing. The partial states need
 *     (P + b*g) * (h/g) * (d_h + 2) * 4 bytes, where
 *     P = min(number of SMs, ceil(b*g*ceil(n_max/64) / 4)); nothing is needed when P is 1;
 *   - the first call on each device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current, so make that first call before any stream capture;
 *   - all calls share the one array, which keeps the last call's contents. The only words that
 *     must start at zero are the per-segment arrival counters: the array is zero when the library
 *     loads, every call that finishes leaves them at zero, and after mqa_get_device_status has
 *     reported MQA_ERR_TIMEOUT the next call clears them first (cudaMemsetAsync, which allocates
 *     nothing). Everything else is written before it is read. Calls that overlap on the GPU (for
 *     instance on two streams at once) race on the array; the caller must order them.
 */
#define MQA_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
#define MQA_NOALLOC_MAX_SEGMENTS 16384u
MQA_API int mqa_decode_attention_noalloc(const mqa_bf16* q, const mqa_bf16* k_cache,
                                         const mqa_bf16* v_cache, const int32_t* seq_lens,
                                         mqa_bf16* out, int b, int h, int g, int d_h, int n_max,
                                         float scale, void* stream);

/*
 * mqa_set_launch_overlap -- let the decode-attention launches on `stream` overlap the kernel
 * immediately ahead of each of them on that stream (programmatic dependent launch). Off by
 * default. The pages have no counterpart; this is a scheduling choice of the library.
 *
 * Why: a launch has a fixed part at both ends -- the pipeline fill before its first tile arrives
 * and, after its last tile, the combine of the pieces of sequences split across CTAs -- during
 * which HBM idles, and its CTAs finish at different times. With overlap on, a launch starts on
 * the SMs that the launch ahead of it has already left and streams its tiles under that launch's
 * drain. This matters for back-to-back decode steps of many layers, where each launch lasts a
 * few hundred microseconds at most.
 *
 * Contract (what the caller guarantees when it turns overlap on for a stream), for every call on
 * the stream and the kernel immediately ahead of it there:
 *   1. that kernel writes none of the call's inputs: q, k_new, v_new, pos, seq_lens, the page
 *      table, and every cache row the call reads other than the rows it appends;
 *   2. that kernel neither reads nor writes the call's outputs: `out` and the cache rows the call
 *      appends.
 * The consecutive layers of one decode step satisfy it (each layer has its own caches and `out`,
 * and all inputs are in place before the first layer is enqueued), and so does any sequence of
 * this library's calls on distinct caches and outputs. A stream that runs mqa_kv_append and then
 * mqa_decode_attention on the same cache does NOT (the append writes a row the attention reads):
 * use the fused mqa_decode_step there. Neither does a call repeated back to back on the same
 * caches and `out`.
 *
 * What the library guarantees in exchange: results are bit for bit those of the same calls with
 * overlap off. A call whose K and V caches together span at most 768 MiB (b*g*n_max rows of
 * d_h elements, counted for both caches) writes early: it never shares its scratch with the
 * launch ahead of it (the stream's workspace has two halves that consecutive launches take in
 * turn). A call over larger caches, and every mqa_decode_attention_noalloc call (one scratch
 * array), reads early but writes nothing -- no output, no scratch, no appended row -- before the
 * kernel ahead has finished. In both cases the launch after a call may start only once the
 * kernel ahead of the call has finished, so no launch runs beside the one two back. The setting
 * applies to the attention, step, paged, fp8, multi-token (h/g * T <= 64) and no-alloc calls on
 * the mma.sync and CUDA-core paths (the forced tcgen05 path and the prefill path never overlap),
 * and to launches captured into a CUDA graph, where it becomes a programmatic edge between
 * consecutive kernel nodes.
 *
 *   stream   cudaStream_t, on the current device (NULL: the legacy default stream)
 *   on       1 to allow overlap, 0 to forbid it
 *
 * Returns MQA_OK, MQA_ERR_INVALID_ARG (on not 0 or 1) or MQA_ERR_CUDA.
 */
MQA_API int mqa_set_launch_overlap(void* stream, int on);

/* A static, human-readable name for a status code. Never returns NULL. */
MQA_API const char* mqa_status_string(int status);

/*
 * Synchronise `stream`, then read and clear the status word latched by kernels on the current
 * device. *status_out receives MQA_OK or the first latched error. Returns MQA_OK, or
 * MQA_ERR_CUDA if the synchronisation or the read failed (for instance after a kernel fault),
 * or MQA_ERR_INVALID_ARG if status_out is NULL.
 */
MQA_API int mqa_get_device_status(void* stream, int* status_out);

/*
 * Diagnostics for MQA_ERR_TIMEOUT: synchronise the current device, then read and clear where the
 * first in-kernel wait that ran out of time gave up. site_out[0] is the wait (0 = none since the
 * last read; 1 producer waiting for a free stage, 2 consumers waiting for a stage's copy, 3 the
 * consumer-wide barrier, 4 the tcgen05 issuer waiting for Q, 5 ... for a stage's copy, 6 ... for P,
 * 7 the softmax warps waiting for S, 8 ... for O before a rescale, 9 ... for a stage's copy,
 * 10 ... for the last O of a segment, 11 the issuer draining its MMAs, 12 the issuer waiting for
 * the softmax warps at exit, 13 the issuer waiting for the P V product that last read an S buffer,
 * 14 the testing stall of mqa_debug_stall); site_out[1] the tile index within the CTA's range, site_out[2] the
 * CTA, site_out[3] the thread. Returns MQA_OK, MQA_ERR_INVALID_ARG (NULL) or MQA_ERR_CUDA.
 */
MQA_API int mqa_debug_timeout_site(int* site_out);

/*
 * Testing hooks for failure detection (process-wide).
 *
 * mqa_debug_set_wait_limit_ns: the limit, in nanoseconds, after which an in-kernel wait gives up
 * and the launch reports MQA_ERR_TIMEOUT (0 restores the default of one second). The waits for a
 * CTA's own copies and MMAs still in flight when it stops keep the one-second limit, so a launch
 * that gave up leaves nothing running. Returns MQA_OK.
 *
 * mqa_debug_stall: with on = 1, the consumer warps of every following attention launch first wait
 * on a barrier that nothing completes, so that wait runs out after the wait limit and the launch
 * reports MQA_ERR_TIMEOUT at site 14 (a flag nothing sets; no fault and no hang). With on = 2 the
 * mma.sync and CUDA-core kernels wait there instead right after a CTA has counted its arrival at a
 * sequence split across CTAs, before any merge, so the launch gives up with arrival counters left
 * non-zero (the tcgen05 kernel stalls at its start, as with 1). on = 0 turns it off. Returns
 * MQA_OK, or MQA_ERR_INVALID_ARG for another value.
 */
MQA_API int mqa_debug_set_wait_limit_ns(uint64_t ns);
MQA_API int mqa_debug_stall(int on);

/* Number of kernels this library has launched in this process (all devices, all streams). */
MQA_API uint64_t mqa_kernel_launch_count(void);

/*
 * Testing hook: force the number of CTAs that split the attention work (0 = automatic choice)
 * and the inner-product path: 0 = automatic (CUDA cores when h/g <= 2 over bf16 caches,
 * mma.sync tensor cores otherwise, and for fp8 caches at every h/g); 1 = CUDA cores (h/g <= 7 only); 2 = mma.sync tensor cores; 3 = tcgen05 tensor cores
 * with tensor-memory accumulators. Process-wide; returns
 * MQA_ERR_INVALID_ARG for a negative CTA count or an unknown path. Results must not depend on
 * either setting beyond rounding.
 */
MQA_API int mqa_debug_override(int num_ctas, int path);

#ifdef __cplusplus
}
#endif

#endif /* MQA_H_ */
