/*
 * librq -- ResidualQuant decode attention over a residual-quantised per-loop KV cache,
 * native to GB300 (sm_103a).  Plain C ABI: device pointers, sizes, a stream handle.
 *
 * The method ("ResidualQuant: KV Cache Quantization for Looped Transformers with 2-Bit
 * Residuals", abstract; rit.work summary, "How each pass's KV cache is reconstructed"):
 * a looped Transformer applies one block L times per token and every loop (pass) makes
 * its own K/V.  For each token, the FINAL loop's K/V is stored as the reference in
 * asymmetric INT4; every other loop l is stored as a residual against the scaled
 * reference,
 *     x_l  ~=  a_l * ref_hat + R^T * deq(res_l),
 * where a_l is the least-squares scale <x_l, ref_hat> / <ref_hat, ref_hat>, R is an
 * orthogonal channel rotation per (layer, kv-head, K/V) and res_l is an asymmetric
 * INT2 (or INT4: loop-wise mixed precision) code of R (x_l - a_l ref_hat).  The current
 * token stays in BF16 until its final loop ends (deferred write); then all its loops are
 * encoded and appended.  Decode attention rebuilds reference and residuals inside the
 * attention computation and never writes decompressed K/V to memory.
 *
 * Conventions for every entry point
 *   - All tensors are caller-owned device memory (except rq_shape / rq_cache structs,
 *     which are host memory read during the call).  The library never allocates, frees
 *     or synchronises; all work is enqueued on `stream` (a cudaStream_t, 0 = legacy
 *     default stream) of the current device.
 *   - fp16 and bf16 tensors are passed as uint16_t pointers holding the raw bits.
 *   - Arguments are validated before anything is enqueued: an invalid call returns a
 *     status and enqueues nothing.  A failed launch returns RQ_ERR_CUDA.  No C++
 *     exception crosses the ABI and the library keeps no mutable global state.
 *
 * Packed cache layout (one layer; kv = 0 for K, 1 for V; d = head_dim, ng = d / 32):
 * one byte array of tile records, [B][Hkv][cap/64] records, one per (sequence, kv-head,
 * 64-token tile), each rq_record_bytes(shape) = 64 * (token-head bytes) long and made of
 * sections, each section 64 rows of one kind, in this order:
 *   reference section:
 *     K codes  [64][d/2]      INT4 reference codes of K
 *     K meta   [64][ng][2]    fp16 (step, offset) per group
 *     V codes  [64][d/2]      INT4 reference codes of V (token-pair order, below)
 *     V meta   [64][ng][2]
 *   then one section per non-final loop l = 0 .. L-2 (b_l = residual bits of loop l):
 *     K codes  [64][d*b_l/8]  residual codes of K
 *     K meta   [64][ng][2]
 *     K a      [64]           fp16 least-squares scale a_l of K
 *     V codes  [64][d*b_l/8]  (token-pair order)
 *     V meta   [64][ng][2]
 *     V a      [64]
 * Row t of a section is token 64 j + t of tile j.  A stage of the decode kernel is one or two
 * contiguous pieces of a record (the reference section and the sections of the loops it
 * needs), so each stage moves with one or two bulk copies.  rot_signs[kv] int8 [Hkv][d]:
 * +-1, R = H_d diag(signs) / sqrt(d).
 * A token's natural code row packs channel i into byte i*b/8 at bit offset (i*b) % 8.
 * K rows store the natural row's 32-bit words group-interleaved: natural word w (the
 * (w % b)-th word of 32-channel group w / b) sits at word (w % b) * (d/32) + w / b.  V rows
 * are stored in token pairs: in pair p (tokens 2p, 2p+1 of the tile) the 32-bit word at
 * position u ^ swz(p) holds 16-bit unit u of token 2p's natural row (low half) and of token
 * 2p+1's (high half), with swz(p) = 8 (p % 4) for 32-unit rows, 8 ((p / 2) % 2) for 16-unit
 * rows and 0 for shorter rows.  Both orders keep each lane's tensor-core operand loads in
 * distinct shared-memory banks.  Capacity must be a multiple of 64.  Groups are 32
 * contiguous channels: original channels for the reference, rotated channels for residuals.
 */
#ifndef RQ_H_
#define RQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RQ_MAX_LOOPS 16

typedef enum {
  RQ_OK = 0,
  RQ_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, range out of bounds   */
  RQ_ERR_UNSUPPORTED = 2, /* head_dim not 64/128, group not 32, bits not 2/4, ...    */
  RQ_ERR_WORKSPACE = 3,   /* workspace missing or smaller than rq_decode_workspace_bytes */
  RQ_ERR_CUDA = 4,        /* a CUDA call or kernel launch failed                     */
  RQ_ERR_INTERNAL = 5
} rq_status;

typedef struct {
  int32_t batch;        /* B                                                          */
  int32_t n_q_heads;    /* Hq, a multiple of n_kv_heads (GQA: query head h reads       */
  int32_t n_kv_heads;   /*     kv-head h / (Hq / Hkv))                                 */
  int32_t head_dim;     /* d: 64 or 128                                               */
  int32_t n_loops;      /* L: 1..16; loop L-1 is the reference                         */
  int32_t group;        /* must be 32                                                  */
  int32_t capacity;     /* tokens per (sequence, kv-head) slot; a multiple of 64       */
  int8_t res_bits[RQ_MAX_LOOPS]; /* residual bits of loop l < L-1: 2 or 4              */
  float softmax_scale;  /* 0 => 1/sqrt(d)                                              */
} rq_shape;

typedef struct {
  uint8_t* data;                /* the tile records (layout above), 256-byte aligned     */
  const int8_t* rot_signs[2];   /* [Hkv][d] per K / V                                    */
} rq_cache;

/* Bytes of one tile record of this shape: 64 x the token-head bytes (0 if invalid). */
size_t rq_record_bytes(const rq_shape* shape);

/* Bytes of one layer's packed cache (all tile records, not rot_signs): per token-head and
 * K/V, d/2 + 4*ng for the reference plus d*b_l/8 + 4*ng + 2 per non-final loop, times
 * B * Hkv * capacity.  Returns 0 for an invalid shape. */
size_t rq_cache_bytes(const rq_shape* shape);

/* Deferred write (rit.work summary, "How each pass's KV cache is reconstructed": the
 * current token's loop states stay in BF16 until the final loop ends, then the
 * compressed cache is written).  Encodes n_new tokens per sequence, all L loops, K and V,
 * every kv-head, and stores them at their cache positions.
 *   kv_new     bf16 element (b, j, kv, l, h, i) at
 *              b*strides[0] + j*strides[1] + kv*strides[2] + l*strides[3] + h*strides[4] + i
 *              (channel stride 1; strides in elements, non-negative)
 *   positions  device int32 [B][n_new]: cache slot of new token j of sequence b; or NULL,
 *              in which case slot = pos_begin + j.  Slots must lie in [0, capacity): a
 *              device-side slot outside that range is skipped (nothing written).
 *   n_new      >= 0 (0: nothing enqueued).
 * The same slot must not be written twice in one call.  Codes, step/offset and a_l follow
 * the header comment's layout; rounding is to nearest even throughout. */
rq_status rq_encode_append(const rq_shape* shape, const rq_cache* cache,
                           const uint16_t* kv_new, const int64_t strides[5],
                           const int32_t* positions, int32_t pos_begin, int32_t n_new,
                           void* stream);

/* Workspace bytes needed by rq_decode_attention / rq_bf16_decode_attention for this
 * shape, loop_count and max_ctx on the current device: a 256-byte header, the split
 * tickets, then the split-KV partials.  After rq_decode_attention completes, the header's
 * first uint32 is 0; it is nonzero if a pipeline wait inside the kernel gave up, a paged
 * call met a bad table entry or a ctx_len lay outside what the call covers.  The outputs of every (sequence, kv-head) whose splits met the
 * fault are then NaN; calls that merge their splits in a separate combine make all outputs
 * NaN.  A caller checks the word, not the outputs. */
size_t rq_decode_workspace_bytes(const rq_shape* shape, int32_t loop_count, int32_t max_ctx);

/* Fused decode attention over the packed cache (rit.work summary, "How each pass's KV
 * cache is reconstructed": reference and residuals are rebuilt in small blocks inside
 * attention, no decompressed K/V is written back).
 *   q          bf16 [B][Hq][loop_count][d]: the queries of loops loop_begin..+loop_count-1
 *   loop_begin, loop_count: 0 <= loop_begin, loop_begin + loop_count <= L, loop_count >= 1.
 *              loop_count = 1 is the causal per-loop call of a real decode step;
 *              loop_count = L supplies all loops' queries at once (the reference tile is
 *              then read once for all loops).
 *   pending_kv bf16 [B][2][loop_count][Hkv][d] (0 = K, 1 = V): the current token's BF16
 *              state of each loop in the call, attended after the cached tokens; or NULL.
 *   ctx_lens   device int32 [B]: cached tokens of each sequence (slots 0..ctx_len-1).
 *   max_ctx    host upper bound of ctx_lens (<= capacity); sizes the split-KV grid.  A
 *              device-side ctx_len above the tokens the grid covers (above max_ctx, as can
 *              happen when a captured graph keeps a fixed max_ctx while ctx_lens advance),
 *              above capacity or negative is not truncated silently: the workspace error
 *              word is set and that sequence's outputs are NaN (see rq_decode_workspace_bytes).
 *   out        bf16 [B][Hq][loop_count][d].  A row with no cached and no pending token
 *              is written as zeros.
 *   ws         device workspace of at least rq_decode_workspace_bytes(...) bytes,
 *              256-byte aligned.  The call clears its head (error word, split tickets) on
 *              the stream and then fills the split records; calls that share a workspace
 *              must not overlap on the GPU.
 * Loop-l queries attend over loop l's rebuilt K/V; scores are scaled by softmax_scale. */
rq_status rq_decode_attention(const rq_shape* shape, const rq_cache* cache,
                              const uint16_t* q, int32_t loop_begin, int32_t loop_count,
                              const uint16_t* pending_kv, const int32_t* ctx_lens,
                              int32_t max_ctx, uint16_t* out, void* ws, size_t ws_bytes,
                              void* stream);

/* Comparison kernel: the same decode attention over an uncompressed BF16 cache,
 *   k, v  bf16 [B][Hkv][L][capacity][d]
 * with every other argument as in rq_decode_attention (Hq / Hkv at most 8). */
rq_status rq_bf16_decode_attention(const rq_shape* shape, const uint16_t* k,
                                   const uint16_t* v, const uint16_t* q, int32_t loop_begin,
                                   int32_t loop_count, const uint16_t* pending_kv,
                                   const int32_t* ctx_lens, int32_t max_ctx, uint16_t* out,
                                   void* ws, size_t ws_bytes, void* stream);

/* Paged cache (rit.work summary, "When ResidualQuant changes the infrastructure plan": the
 * pages' integration keeps the serving engine's paged KV cache; this is its block-table
 * form).  A page holds 64 consecutive tokens of one sequence for every kv-head: in paged
 * mode the tile records are [n_pages][Hkv] instead of [B][Hkv][cap/64], each the same record
 * as above.  Tokens 64j..64j+63 of sequence b live in physical page
 * block_table[b * max_pages + j].  shape->capacity must equal 64 * max_pages (the logical
 * capacity of a sequence).  The table is read on the device: an entry outside
 * [0, n_pages) is never dereferenced -- the encode skips that token, the decode reads page 0
 * instead and flags the workspace error word (the affected outputs NaN). */
typedef struct {
  const int32_t* block_table;  /* device int32 [B][max_pages]                         */
  int32_t max_pages;           /* table columns: logical pages per sequence            */
  int32_t n_pages;             /* physical pages (records per kv-head)                 */
} rq_paging;

/* Bytes of one layer's paged cache with n_pages physical pages (0 for an invalid shape). */
size_t rq_paged_cache_bytes(const rq_shape* shape, int32_t n_pages);

/* rq_encode_append on a paged cache: positions are logical token positions of each
 * sequence (< capacity); the slot is found through the block table. */
rq_status rq_paged_encode_append(const rq_shape* shape, const rq_cache* cache,
                                 const rq_paging* paging, const uint16_t* kv_new,
                                 const int64_t strides[5], const int32_t* positions,
                                 int32_t pos_begin, int32_t n_new, void* stream);

/* rq_decode_attention on a paged cache (same arguments, same workspace size, same
 * results bit for bit as on a contiguous cache holding the same tokens). */
rq_status rq_paged_decode_attention(const rq_shape* shape, const rq_cache* cache,
                                    const rq_paging* paging, const uint16_t* q,
                                    int32_t loop_begin, int32_t loop_count,
                                    const uint16_t* pending_kv, const int32_t* ctx_lens,
                                    int32_t max_ctx, uint16_t* out, void* ws, size_t ws_bytes,
                                    void* stream);

/* Decode attention without a caller-provided workspace, for callers that cannot allocate
 * device memory: e.g. a plug-in whose host framework owns every device allocation and hands
 * it only input and output tensors, or a C caller that must not allocate once it has
 * started.  (The method's pages have no counterpart: this is an interface choice.)
 * The split-KV scratch lives in a fixed device array of rq_decode_noalloc_scratch_bytes()
 * bytes (32 MiB) inside the library; every GPU that loads the library holds that array until
 * the process exits.  Arguments are as in rq_decode_attention without ws / ws_bytes.
 *   - A call whose scratch need (rq_decode_workspace_bytes) exceeds the array returns
 *     RQ_ERR_WORKSPACE and enqueues nothing.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.
 *   - No allocation of any kind: no cudaMalloc, cudaFree or allocating library routine.
 *   - All calls share the one array and it keeps the last call's contents: calls whose
 *     executions overlap on the GPU (other streams, other host threads) race on it, so
 *     serialise them.  Each call clears what must start at zero itself. */
size_t rq_decode_noalloc_scratch_bytes(void);
rq_status rq_decode_attention_noalloc(const rq_shape* shape, const rq_cache* cache,
                                      const uint16_t* q, int32_t loop_begin, int32_t loop_count,
                                      const uint16_t* pending_kv, const int32_t* ctx_lens,
                                      int32_t max_ctx, uint16_t* out, void* stream);

/* Human-readable name of a status. */
/* Serving step support (rit.work summary, "How each pass's KV cache is reconstructed": the
 * current token's loops are encoded once its final loop ends, then it joins the cache).
 * Adds n to every ctx_lens[b] on the device, capped at capacity, so that a captured CUDA graph
 * of one decode step -- the per-loop decode calls, rq_encode_append with positions = ctx_lens
 * (n_new = 1: the new token goes to slot ctx_len) and this call -- can be replayed token after
 * token.  ctx_lens: device int32 [batch]; n >= 0. */
rq_status rq_advance_ctx(int32_t* ctx_lens, int32_t batch, int32_t n, int32_t capacity,
                         void* stream);

const char* rq_status_str(rq_status status);

#ifdef __cplusplus
}
#endif

#endif /* RQ_H_ */
