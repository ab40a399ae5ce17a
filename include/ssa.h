/*
 * ssa.h -- C ABI of the content-routed sparse attention library (libssa.so).
 *
 * The method (superlinear release post, geeks.co.kr/post/2077, key-idea
 * section; SubQ SSA pages, stork.ai "SubQ AI: 1000x compute"): the context
 * is cut into spans of about sqrt(L) tokens; each query scores the span
 * summaries, keeps its top-k spans, and runs exact softmax attention over
 * the tokens of those spans.  The pages leave the router open ("learned
 * routing"); this library fixes it as follows:
 *   summary_j = mean of the keys of span j             (fp32)
 *   score_j   = q . summary_j, unscaled                (fp32)
 *   candidates of a query at position t: the complete spans 0 .. l-1,
 *     l = floor(t / S) being the query's own (local) span
 *   selection = the k best candidates under (score desc, index asc)
 *   attended tokens = the selected spans plus [l*S, t] (causal local span)
 *   O = softmax(scale * q K^T) V over the attended tokens, lse = log-sum-exp
 *
 * Conventions shared by every entry point
 *   Layouts (row-major, contiguous, element type = params.dtype):
 *     Q prefill [B, Hq, n_q, d]      query i sits at position q_pos0 + i
 *     Q decode  [B, Hq, d]           one query per head at position `pos`
 *     K, V      [B, Hkv, L_cap, d]   the cache; rows 0 .. L-1 are valid
 *     summ      [B, Hkv, ns_cap, d]  fp32, ns_cap = ceil(L_cap / S)
 *     sel       [B, Hq, n_q, topk]   int32 span indices, ascending, padded
 *                                    with -1 (decode: n_q = 1)
 *     O         like Q; lse [B, Hq, n_q] fp32 (natural log)
 *   Query head h reads kv-head h / (Hq / Hkv) (contiguous GQA groups).
 *   Pointers: every tensor argument is a device pointer owned by the
 *   caller; the library allocates no memory and keeps no state between
 *   calls other than per-device attributes read once.
 *   Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *   default stream).  Every call only enqueues work on it and returns
 *   without synchronising the host.
 *   Errors: argument errors are detected on the host and returned before
 *   anything is enqueued; a failed launch returns SSA_ERR_CUDA.  Errors the
 *   GPU detects (a sel entry that is not a candidate of its query, a wait
 *   that exceeded its bound) are OR-ed into the first 4 bytes of the
 *   workspace; read them with ssa_workspace_error after the stream is done.
 *   No kernel traps or asserts.
 *   Workspace: `ws` is caller-owned device memory of at least
 *   ssa_workspace_size(...) bytes, 256-byte aligned, zeroed once before its
 *   first use.  Its first 256 bytes are a header whose first uint32 is the
 *   sticky error record; the rest is scratch that one call may overwrite, so
 *   calls that share a workspace must be ordered on one stream.
 *   Supported: d in {64, 128}; S >= 1; 1 <= topk <= 64; Hq a multiple of
 *   Hkv with Hq / Hkv <= 16; dtype fp32, bf16 or fp16.  Other values return
 *   SSA_ERR_UNSUPPORTED.
 */
#ifndef SSA_H
#define SSA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSA_API __attribute__((visibility("default")))
#else
#define SSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSA_OK = 0,
  SSA_ERR_INVALID_ARG = 1, /* null pointer, negative size, range outside the cache, ... */
  SSA_ERR_UNSUPPORTED = 2, /* valid but not implemented (d, topk, group size, dtype) */
  SSA_ERR_WORKSPACE = 3,   /* ws is NULL, misaligned or smaller than required */
  SSA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  SSA_ERR_DEVICE = 5,      /* the GPU flagged an error in the workspace record */
  SSA_ERR_IO = 6           /* a snapshot file could not be opened, read or written, or is not one */
} ssa_status;

typedef enum { SSA_F32 = 0, SSA_BF16 = 1, SSA_F16 = 2 } ssa_dtype;

/* Operation selector of ssa_workspace_size. */
typedef enum { SSA_OP_ROUTE = 0, SSA_OP_DECODE = 1, SSA_OP_PREFILL = 2, SSA_OP_ROUTE_GROUP = 3 } ssa_op;

/* Bits of the device error record (first uint32 of a workspace). */
#define SSA_DEVERR_BAD_SELECTION 0x1u /* sel entry not in -1 .. l-1, not ascending, or repeated */
#define SSA_DEVERR_WAIT_TIMEOUT 0x2u  /* a bounded wait on a barrier gave up */
#define SSA_DEVERR_OVERFLOW 0x4u      /* a work list outgrew the space sized for it */

typedef struct {
  int32_t B;      /* batch */
  int32_t Hq;     /* query heads */
  int32_t Hkv;    /* key/value heads; Hq % Hkv == 0 */
  int32_t d;      /* head dimension */
  int64_t L;      /* valid cache length: rows 0 .. L-1 of K and V hold data */
  int64_t L_cap;  /* rows per (b, kv-head) in K and V (head stride L_cap * d); 0 means L */
  int32_t S;      /* span length */
  int32_t topk;   /* spans kept per query (besides the local span) */
  float scale;    /* attention scale; 0 means 1 / sqrt(d) */
  int32_t dtype;  /* ssa_dtype of Q, K, V and O */
} ssa_params;

/*
 * Span summaries (superlinear post, key-idea section: the spans that get
 * scored; the summary itself is fixed by the specification as the mean).
 * Writes summ[b, kvh, j, :] = (1 / n_j) * sum of K[b, kvh, t, :] over the
 * n_j = min(S, L - j*S) valid tokens t of span j, for every span j in
 * [span_begin, span_end) (fp32 accumulation, fp32 result).  Other rows of
 * summ are left untouched, so a chunked prefill calls this once per chunk
 * for the spans the chunk completed.
 * Requires 0 <= span_begin <= span_end <= ceil(L / S).
 */
SSA_API int ssa_build_summaries(const ssa_params* p, const void* K, int64_t span_begin,
                        int64_t span_end, float* summ, void* stream);

/*
 * Routing: span scores and top-k selection (superlinear post, key-idea
 * section: score the O(L^0.5) candidate spans and keep the top k).
 * For each query row (b, h, i) at position t = q_pos0 + i with local span
 * l = floor(t / S): scores q . summ[b, h / g, j, :] (fp32) for j < l and
 * writes the min(l, topk) best under (score desc, j asc) to sel[b, h, i, :]
 * in ascending j, then -1 up to topk.  sel_score (nullable, [B, Hq, n_q,
 * topk] fp32) receives the score of each written span (NaN beside a -1).
 * Summaries of spans 0 .. floor((q_pos0 + n_q - 1) / S) - 1 must be built.
 * Requires n_q >= 0, q_pos0 >= 0, q_pos0 + n_q <= L.
 * A chunk (n_q > 1) of bf16 / fp16 queries is scored on the tensor cores
 * against a three-way 16-bit split of the fp32 summaries kept in ws; ws may
 * be NULL when ssa_workspace_size(p, n_q, SSA_OP_ROUTE) is 0 (decode, fp32).
 */
SSA_API int ssa_route(const ssa_params* p, const void* Q, int64_t n_q, int64_t q_pos0,
              const float* summ, int32_t* sel, float* sel_score, void* ws, size_t ws_bytes,
              void* stream);

/*
 * Group-shared routing for grouped-query attention: one selection per
 * (b, kv-head, query), used by all g = Hq / Hkv query heads of the group.
 * The pages leave the router open (superlinear post, key-idea section: each
 * query keeps the top k of the candidate spans); this variant scores span j
 * of kv-head h for the group as score_j = sum over its query heads hq of
 * q_hq . summ[b, h, j, :] (fp32), keeps the k best under (score desc, j asc)
 * over the same candidates (the complete spans before the query's own), and
 * writes that row to sel[b, hq, i, :] for every head hq of the group (and
 * the scores to sel_score when not NULL).  Arguments, layouts and
 * requirements as for ssa_route; ws must hold
 * ssa_workspace_size(p, n_q, SSA_OP_ROUTE_GROUP) bytes.  The selections then
 * go to ssa_attend_decode / ssa_attend_prefill unchanged; with all heads of
 * a group on the same spans, decode streams k spans plus the local span per
 * kv-head.
 */
SSA_API int ssa_route_group(const ssa_params* p, const void* Q, int64_t n_q, int64_t q_pos0,
                            const float* summ, int32_t* sel, float* sel_score, void* ws,
                            size_t ws_bytes, void* stream);

/*
 * Decode attention for one query per head at position `pos` (superlinear
 * post, key-idea section: token-level attention inside the chosen spans;
 * SubQ SSA page: exact attention over the content-selected subset).
 * sel is [B, Hq, topk] as written by ssa_route with n_q = 1, q_pos0 = pos.
 * Each query group of one kv-head streams the union of its heads' selected
 * spans once, split across the GPU, and a log-sum-exp merge combines the
 * pieces in ascending span order.  Writes O [B, Hq, d] (params.dtype) and,
 * if lse is not NULL, lse [B, Hq] (fp32).
 * Requires 0 <= pos < L.
 */
SSA_API int ssa_attend_decode(const ssa_params* p, const void* Q, int64_t pos, const void* K,
                      const void* V, const int32_t* sel, void* O, float* lse, void* ws,
                      size_t ws_bytes, void* stream);

/*
 * One whole decode step: ssa_route with n_q = 1 at q_pos0 = pos, then
 * ssa_attend_decode on its selections (superlinear post, key-idea section:
 * each new token scores the candidate spans, keeps the top k and attends
 * their tokens plus its own span).  Same arguments, layouts and results as
 * those two calls in sequence: sel [B, Hq, topk] receives the selections,
 * O [B, Hq, d] and lse [B, Hq] (nullable) the outputs; ws as for
 * ssa_attend_decode (ssa_workspace_size(p, 1, SSA_OP_DECODE) bytes).
 * On the 16-bit fast path the step is three kernel launches instead of the
 * separate calls' four: the route kernel's cluster also builds the attend
 * plan, then the split attention and the log-sum-exp merge run.  Other
 * shapes (fp32) run the two calls' kernels in sequence.
 * On the 16-bit fast path Q, sel, O and lse may also be page-locked host
 * memory mapped into the device's address space (cudaHostAlloc or
 * cudaHostRegister under unified addressing): the route kernel reads Q once
 * and keeps a copy in ws for the attention, and sel, O and lse are written
 * in place, so a step needs no separate copies.  Any other host pointer
 * there is SSA_ERR_INVALID_ARG.
 * Requires 0 <= pos < L; summaries of spans 0 .. floor(pos / S) - 1 built.
 */
SSA_API int ssa_decode_step(const ssa_params* p, const void* Q, int64_t pos, const float* summ,
                            const void* K, const void* V, int32_t* sel, void* O, float* lse,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * One whole decode step with group-shared selection: ssa_route_group
 * (n_q = 1) followed by ssa_attend_decode, in three launches (the router
 * sums each group's queries in fp32 in head order, as ssa_route_group does,
 * scores the sum, writes the group's selection to all g heads' sel rows and
 * builds the attend plan in its cluster; then the attention and the merge).
 * The selections are bit-identical to the two calls; O and lse agree to
 * rounding, since the step splits the group's spans into smaller work items
 * (a group-shared union is k + 1 spans, not up to g k + 1).  Arguments as for
 * ssa_decode_step; ws as for ssa_attend_decode (ssa_workspace_size(p, 1,
 * SSA_OP_DECODE) bytes; no group-routing workspace is needed).  Q, sel, O
 * and lse may be mapped page-locked host memory.  16-bit types and the
 * shapes of the fast decode path only (ssa_attend_path(p, 1, SSA_OP_DECODE)
 * == SSA_PATH_FAST); otherwise SSA_ERR_UNSUPPORTED.
 */
SSA_API int ssa_decode_step_group(const ssa_params* p, const void* Q, int64_t pos, const float* summ,
                                  const void* K, const void* V, int32_t* sel, void* O, float* lse,
                                  void* ws, size_t ws_bytes, void* stream);

/*
 * Chunked-prefill attention for n_q queries at positions q_pos0 .. q_pos0 +
 * n_q - 1 (superlinear post: chunked prefill against the kept cache; the
 * attention itself as for ssa_attend_decode).  Work is dispatched span-major:
 * the (query, head) pairs that chose a span are gathered into tiles that
 * stream the span's keys and values once per tile.  Writes O [B, Hq, n_q, d]
 * (params.dtype) and, if lse is not NULL, lse [B, Hq, n_q] (fp32).
 * Requires n_q >= 0, q_pos0 >= 0, q_pos0 + n_q <= L.
 */
SSA_API int ssa_attend_prefill(const ssa_params* p, const void* Q, int64_t n_q, int64_t q_pos0,
                       const void* K, const void* V, const int32_t* sel, void* O, float* lse,
                       void* ws, size_t ws_bytes, void* stream);

/* Size of the library's own decode scratch block, one per device (8 MiB). */
#define SSA_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * ssa_attend_decode without a caller-supplied workspace.  The method's
 * pages have no counterpart to this call: it is an interface convenience,
 * and the attention it computes is exactly that of ssa_attend_decode.
 *
 * It serves callers that cannot allocate device memory at the point of the
 * call, such as a plugin whose host runtime owns every device allocation,
 * or a decode loop that must never reach an allocator.  The scratch is a
 * block of SSA_NOALLOC_SCRATCH_BYTES that the library defines as static
 * device memory; it exists once per device from the moment the library's
 * device code is loaded.  No call allocates or frees anything.
 *
 * Arguments, layouts and the returned status are those of
 * ssa_attend_decode, plus:
 *   scratch  nullable; receives the device address of the block, whose
 *            first uint32 is the sticky device error record, as in any
 *            workspace.  Read it with ssa_workspace_error(*scratch, ...).
 *            The library keeps ownership.
 * Limit: if ssa_workspace_size(p, 1, SSA_OP_DECODE) exceeds
 *   SSA_NOALLOC_SCRATCH_BYTES, returns SSA_ERR_WORKSPACE and enqueues
 *   nothing; use ssa_attend_decode with a workspace of that size instead.
 * Set-up: every call looks up the block's address in the current device's
 *   current context (a host-side lookup); the first call in a context also
 *   enqueues a clear of its error record on `stream`.  Make that first call
 *   before any stream capture begins, and again after cudaDeviceReset (the
 *   device's next context gets its own block and its own first call).
 * Races: every call on one device shares the block.  Calls that can overlap
 *   in time (two streams, two host threads) corrupt each other's results and
 *   error record; keep them on one stream.
 */
SSA_API int ssa_attend_decode_noalloc(const ssa_params* p, const void* Q, int64_t pos,
                                      const void* K, const void* V, const int32_t* sel, void* O,
                                      float* lse, void** scratch, void* stream);

/*
 * The 8-bit cache (SubQ release post, geeks.co.kr/post/2077, limitations
 * and quantisation plan: fp16 only so far, 8-bit / 4-bit K / V coming so
 * that a 1M-token cache fits a 24 GB card).  The pages fix no scheme; this
 * library uses symmetric 8-bit rows, one fp32 scale per (b, kv-head, token):
 *   s = max_i |x_i| / 127,  q_i = clamp(rint(x_i / s), -127, 127), 0 if s == 0
 * in fp32 (IEEE division, round to nearest even); a row's dequantised value
 * is q_i * s.  Summaries stay fp32 (the mean of the dequantised keys), so
 * routing is ssa_route / ssa_route_group on them, unchanged.
 * Layouts (params.L_cap must be a multiple of 32; d = 128 for attention):
 *   Kq [B, Hkv, L_cap, d]            int8, row-major
 *   Vq [B, Hkv, L_cap / 32, d, 32]   int8: each 32-token tile stored d-major;
 *        in a tile's d-row of 32 bytes, byte 8 c + e (c = 0..3, e = 0..7)
 *        holds token 16 * (e / 4) + (2c, 2c+1, 2c+8, 2c+9)[e % 4] of the tile
 *   Ks, Vs [B, Hkv, L_cap]           fp32 scales
 * Every pointer is 16-byte aligned device memory owned by the caller.
 */

/*
 * Quantises rows [t_begin, t_end) of every (b, kv-head) of K and V (layouts
 * of the conventions above, element type params.dtype) into Kq, Ks, Vq, Vs.
 * Other rows are untouched, so a decode loop quantises each new token and a
 * chunked prefill each chunk.  Requires 0 <= t_begin <= t_end <= L.
 */
SSA_API int ssa_quantize_kv(const ssa_params* p, const void* K, const void* V, int64_t t_begin,
                            int64_t t_end, int8_t* Kq, float* Ks, int8_t* Vq, float* Vs, void* stream);

/*
 * ssa_build_summaries over the 8-bit keys: summ[b, kvh, j, :] = mean over
 * span j's valid tokens of Kq * Ks (fp32), for spans [span_begin, span_end).
 */
SSA_API int ssa_build_summaries_q8(const ssa_params* p, const int8_t* Kq, const float* Ks,
                                   int64_t span_begin, int64_t span_end, float* summ, void* stream);

/*
 * ssa_attend_decode over the 8-bit cache: the same selections, work split
 * and merge, with K[t] = Kq[t] * Ks[t] and V[t] = Vq[t] * Vs[t].  Q and O are
 * bf16 or fp16 (params.dtype), d = 128.  The products run in fp16 (8-bit
 * values convert exactly; Q is rounded to fp16, so |q| must stay below
 * 65504) with fp32 accumulation.  ws as for ssa_attend_decode
 * (ssa_workspace_size(p, 1, SSA_OP_DECODE) bytes).  Requires 0 <= pos < L.
 */
SSA_API int ssa_attend_decode_q8(const ssa_params* p, const void* Q, int64_t pos, const int8_t* Kq,
                                 const float* Ks, const int8_t* Vq, const float* Vs, const int32_t* sel,
                                 void* O, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * One whole decode step over the 8-bit cache: ssa_route with n_q = 1 at
 * q_pos0 = pos, then ssa_attend_decode_q8 on its selections, in three kernel
 * launches (the route kernel's cluster also builds the attend plan).  Same
 * arguments, layouts, requirements and results as those two calls in
 * sequence: summ are the fp32 summaries (ssa_build_summaries_q8), sel
 * [B, Hq, topk] receives the selections, O [B, Hq, d] and lse [B, Hq]
 * (nullable) the outputs.  Returns SSA_ERR_UNSUPPORTED where
 * ssa_attend_decode_q8 does.  Q, sel, O and lse may be mapped page-locked
 * host memory as for ssa_decode_step.
 */
SSA_API int ssa_decode_step_q8(const ssa_params* p, const void* Q, int64_t pos, const float* summ,
                               const int8_t* Kq, const float* Ks, const int8_t* Vq, const float* Vs,
                               int32_t* sel, void* O, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * The 4-bit cache (SubQ release post, geeks.co.kr/post/2077, quantisation
 * plan: its 4-bit half).  Symmetric rows, one fp32 scale per (b, kv-head,
 * token): s = max_i |x_i| / 7, q_i = clamp(rint(x_i / s), -7, 7) in fp32
 * (IEEE division, round to nearest even; q = 0 when s == 0), each code
 * stored as the 4-bit field q + 8.  d = 128 and L_cap a multiple of 32.
 * Layouts (32-bit words, little-endian; a 32-token tile of K or of V is one
 * contiguous block of 512 words):
 *   Kq4 [B, Hkv, L_cap / 32][J < 4][tok < 32][c < 4] words: token tok of the
 *       tile, dimensions d = 32 J + 8 c + e, e < 8
 *   Vq4 [B, Hkv, L_cap / 32][d < 128][c < 4] words: dimension d of the tile's
 *       tokens 2 c + (0, 1, 8, 9, 16, 17, 24, 25)[e], e < 8
 *   element e of a word at bits 4 (e / 2) + 16 (e % 2)
 *   Ks, Vs [B, Hkv, L_cap] fp32 scales
 * Kq4 and Vq4 are B * Hkv * L_cap * 64 bytes each.
 */

/*
 * Quantises rows [t_begin, t_end) of K and V into the 4-bit cache.  Tiles
 * the range only partly covers keep their other tokens' codes; calls that
 * touch the same 32-token tile must not overlap in time.
 */
SSA_API int ssa_quantize_kv4(const ssa_params* p, const void* K, const void* V, int64_t t_begin, int64_t t_end,
                             void* Kq4, float* Ks, void* Vq4, float* Vs, void* stream);

/*
 * ssa_build_summaries over the 4-bit keys: summ[b, kvh, j, :] = mean over
 * span j's valid tokens of q * s (fp32), for spans [span_begin, span_end).
 */
SSA_API int ssa_build_summaries_q4(const ssa_params* p, const void* Kq4, const float* Ks, int64_t span_begin,
                                   int64_t span_end, float* summ, void* stream);

/*
 * ssa_attend_decode over the 4-bit cache: the same selections, work split
 * and merge, with K[t] = q_K[t] * Ks[t] and V[t] = q_V[t] * Vs[t].  Q and O
 * are bf16 or fp16, d = 128; the products run in fp16 (4-bit codes convert
 * exactly; Q is rounded to fp16, so |q| must stay below 65504) with fp32
 * accumulation.  ws as for ssa_attend_decode.  Requires 0 <= pos < L.
 */
SSA_API int ssa_attend_decode_q4(const ssa_params* p, const void* Q, int64_t pos, const void* Kq4, const float* Ks,
                                 const void* Vq4, const float* Vs, const int32_t* sel, void* O, float* lse,
                                 void* ws, size_t ws_bytes, void* stream);

/*
 * One whole decode step over the 4-bit cache, as ssa_decode_step_q8 is for
 * the 8-bit one (three launches; Q, sel, O and lse may be mapped page-locked
 * host memory).  summ are the fp32 summaries (ssa_build_summaries_q4).
 */
SSA_API int ssa_decode_step_q4(const ssa_params* p, const void* Q, int64_t pos, const float* summ,
                               const void* Kq4, const float* Ks, const void* Vq4, const float* Vs, int32_t* sel,
                               void* O, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * Cache snapshots (superlinear release post, geeks.co.kr/post/2077, "why
 * this matters": the cache is kept instead of re-processing the context, in
 * memory for instant replies and saved to / restored from disk per session).
 * A snapshot holds the first n_tokens rows of every (b, kv-head) of K and V
 * and the summaries of the n_tokens / S complete spans, so that a restored
 * session routes and attends exactly as the saved one did.
 *
 * File format (little-endian), the header below followed by the payload:
 *   K rows   [B][Hkv][n_tokens][d]  element type dtype
 *   V rows   [B][Hkv][n_tokens][d]  element type dtype
 *   summ     [B][Hkv][n_summ][d]    fp32, n_summ = floor(n_tokens / S)
 * There is no checksum; the file size must equal 64 + payload_bytes.
 */
#define SSA_SNAPSHOT_MAGIC "SSAKVSN1"
#define SSA_SNAPSHOT_VERSION 1u

typedef struct {
  char magic[8];          /* SSA_SNAPSHOT_MAGIC, not NUL-terminated */
  uint32_t version;       /* SSA_SNAPSHOT_VERSION */
  int32_t dtype;          /* ssa_dtype of K and V */
  int32_t B, Hkv, d, S;   /* as in ssa_params */
  int64_t n_tokens;       /* cache rows per (b, kv-head) in the file */
  int64_t n_summ;         /* summaries per (b, kv-head): n_tokens / S */
  uint64_t payload_bytes; /* bytes after the header */
  uint8_t reserved[8];    /* zero */
} ssa_snapshot_header;    /* 64 bytes */

/*
 * Writes a snapshot of rows 0 .. n_tokens-1 of K and V (device, the layouts
 * of the conventions above, head stride L_cap * d) and of summ rows
 * 0 .. n_tokens / S - 1 (device) to the file `path`, replacing it.
 * `staging` is caller-owned host memory of staging_bytes (page-locked for
 * speed; at least 2 * d * 4 bytes, a few tens of MiB recommended): the copy
 * runs in chunks of staging_bytes / 2, device-to-host on `stream` into one
 * half while the other half is written to the file.  The copies follow
 * whatever was enqueued on `stream` before.  Unlike every other entry
 * point, this call returns only when the file is complete (or on error).
 * It allocates no device memory; it creates two CUDA events for the
 * hand-off between the halves and destroys them before returning.
 * Requires 0 <= n_tokens <= L (params.L).
 * Returns SSA_ERR_INVALID_ARG for bad arguments (checked before anything
 * touches the GPU or the file), SSA_ERR_IO when the file cannot be
 * written, SSA_ERR_CUDA when a copy fails.
 */
SSA_API int ssa_snapshot_save(const ssa_params* p, int64_t n_tokens, const void* K, const void* V,
                              const float* summ, const char* path, void* staging, size_t staging_bytes,
                              void* stream);

/*
 * Restores a snapshot written by ssa_snapshot_save into K, V and summ
 * (device, caller-owned, laid out by `p`): rows 0 .. n_tokens-1 of every
 * (b, kv-head) of K and V and summ rows 0 .. n_tokens / S - 1.  Other rows
 * are left untouched.  *n_tokens (nullable) receives the row count; the
 * caller then decodes with params.L = n_tokens.  The file's B, Hkv, d, S
 * and dtype must equal p's and n_tokens must fit L_cap (params.L_cap, or L
 * when 0); otherwise returns SSA_ERR_IO and writes nothing to the device.
 * `staging` and `stream` as for ssa_snapshot_save (host-to-device copies
 * overlap the file reads); returns when the copies are complete.
 */
SSA_API int ssa_snapshot_load(const ssa_params* p, const char* path, void* K, void* V, float* summ,
                              int64_t* n_tokens, void* staging, size_t staging_bytes, void* stream);

/*
 * Reads and checks the header of a snapshot file (host only, no GPU):
 * SSA_OK when the magic, version, reserved bytes, payload size and file
 * size agree, else SSA_ERR_IO.  *out (nullable) receives the header.
 */
SSA_API int ssa_snapshot_read_header(const char* path, ssa_snapshot_header* out);

/* Implementation an attention call takes (ssa_attend_path). */
typedef enum {
  SSA_PATH_INVALID = 0, /* the parameters are invalid or unsupported */
  SSA_PATH_FAST = 1,    /* 16-bit fast path: split / span-major tiles on the tensor cores */
  SSA_PATH_ROWS = 2     /* one warp per query row on the CUDA cores (fp32, or shapes the fast path does not take) */
} ssa_path;

/*
 * Which implementation ssa_attend_decode (op = SSA_OP_DECODE; also
 * ssa_decode_step) or ssa_attend_prefill (op = SSA_OP_PREFILL, n_q queries)
 * takes for these parameters; SSA_PATH_INVALID for other ops or when the
 * parameters would be rejected.  Both paths compute the same attention (the
 * row kernel is slower); this lets a caller see the choice without timing
 * it.  Host only, no GPU.  The prefill fast path needs bf16 / fp16, d in
 * {64, 128}, 128 divisible by Hq / Hkv and B * Hq * n_q < 2^25; the decode
 * fast path needs bf16 / fp16 and B * Hkv <= 1024.
 */
SSA_API int ssa_attend_path(const ssa_params* p, int64_t n_q, int op);

/*
 * Bytes of workspace the operation needs for n_q queries (n_q is ignored
 * for SSA_OP_DECODE), or 0 when the parameters are invalid or unsupported
 * and no workspace is needed (SSA_OP_ROUTE may legitimately return 0).
 * Never fails loudly: validate with the entry point itself.
 */
SSA_API size_t ssa_workspace_size(const ssa_params* p, int64_t n_q, int op);

/*
 * Reads and clears the device error record at the start of ws: waits for
 * `stream`, copies the record to the host, zeroes it, and returns SSA_OK or
 * SSA_ERR_DEVICE; *bits (nullable) receives the SSA_DEVERR_* bits.  This is
 * the one entry point that synchronises the host.
 */
SSA_API int ssa_workspace_error(void* ws, uint32_t* bits, void* stream);

/*
 * Diagnostic with no counterpart in the pages: one thread waits limit_ns
 * nanoseconds (at most 1 s) on a barrier that nothing completes, as the
 * library's kernels wait for their bulk copies and tensor-core work, gives
 * up, ORs SSA_DEVERR_WAIT_TIMEOUT into the error record of ws (ws_bytes >=
 * 256) and returns; no copy or tensor-core work is in flight.  It shows that
 * a wait that runs out comes back as a status the host reads
 * (ssa_workspace_error) and leaves the context usable.  SSA_ERR_INVALID_ARG
 * above 1 s; SSA_ERR_WORKSPACE for a missing or short ws.
 */
SSA_API int ssa_selftest_wait_timeout(uint64_t limit_ns, void* ws, size_t ws_bytes, void* stream);

/* Static text for a status code (never NULL). */
SSA_API const char* ssa_status_string(int status);

/* Library version as major * 10000 + minor * 100 + patch. */
SSA_API int ssa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSA_H */
