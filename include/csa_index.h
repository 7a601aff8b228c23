/*
 * csa_index.h — C ABI of the CSA indexer hot path for GB300 (sm_103a).
 *
 * What the library computes (FlashMemory-DeepSeek-V4, "Retriever architecture"
 * and "compressed_k format"): for every query row b and every visible record n
 * of a paged compressed-K cache,
 *
 *     k_n[d]   = e4m3(rec_n[d]) * scale_n          d < 128, scale_n = fp32 at bytes 128..131
 *     logit_bn = sum_h relu(k_n . q_b[h]) * fused_w_b[h]
 *     score_bn = sigmoid(logit_bn)                 in [0, 1]
 *
 * and keeps the top-k records of each query ("Two-level recall algorithm",
 * Level 2: the top-512 is taken over the whole history or, with non-resident
 * logits masked to -inf, over a resident page subset).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer handed to a compute entry point is DEVICE memory owned by the
 *   caller, except the args struct itself, which is read on the host during the
 *   call only. The library never allocates, frees, synchronises or reads device
 *   data on the host; all work is enqueued on `stream` (a cudaStream_t passed as
 *   void*, NULL = legacy default stream). The only state it keeps is a one-time
 *   per-device kernel attribute set-up (dynamic shared memory size) and the
 *   device's SM count; both are taken on the first call on a device and kept for
 *   the life of the process (as is the built-in scratch address of
 *   csa_index_score_topk_fused_static). The library must therefore not be used on
 *   a device across cudaDeviceReset: the kept state would describe the old
 *   context.
 * - Calls are re-entrant and capturable in a CUDA graph as long as their
 *   workspaces do not overlap while in flight.
 * - Host-detectable errors return a csa_status and launch nothing.
 *   Data-dependent errors found on the device never trap: they OR a CSA_DEV_*
 *   bit into *dev_status (when given) and the offending page or query is left
 *   out of the result.
 *
 * Cache geometry ("compressed_k format"): a record is 132 bytes, 128 e4m3 bytes
 * (OCP FP8 E4M3, the `float8_e4m3fn` variant: bias 7, max 448, S.1111.111 = NaN)
 * followed by a little-endian IEEE fp32 scale. 64 records form a page; pages
 * sit at `page_stride_bytes` apart (>= 64*132, a multiple of 16, so allocator
 * padding is allowed, as the geometry guard of the BatchGen #153 commit log asks
 * for).
 *
 * Lengths (`q_len`) count compressed records, not tokens (BatchGen #153 commit
 * log: passing raw token counts to the c4 indexer read 4x out of bounds).
 */
#ifndef CSA_INDEX_H
#define CSA_INDEX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Raised whenever an entry point, a struct layout or the meaning of an argument changes.
 * 2: csa_index_logits, csa_index_write_keys and the Level-1 recall entry points; 128 heads
 *    in the score and logit modes; a larger fused-path workspace (num_q + 2 row offsets). */
#define CSA_ABI_VERSION 4

#define CSA_HEAD_DIM 128        /* D: e4m3 bytes per record                         */
#define CSA_NUM_HEADS 64        /* H of the Level-2 indexer                         */
#define CSA_RECORD_BYTES 132    /* D + 4-byte fp32 scale                            */
#define CSA_PAGE_RECORDS 64     /* records per page                                 */
#define CSA_PAGE_BYTES 8448     /* 64 * 132                                         */
#define CSA_MAX_K 1024          /* largest top-k supported                          */
#define CSA_MAX_CTAS 1024       /* upper bound on the persistent grid, sizes slots  */

typedef enum csa_status {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, k out of [1, CSA_MAX_K] ...   */
  CSA_ERR_UNSUPPORTED = 2,   /* head_dim != 128, num_heads other than 64 (or 128 where
                                allowed), too many SMs                                       */
  CSA_ERR_ALIGNMENT = 3,     /* a pointer or stride breaks the alignment stated below       */
  CSA_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than csa_index_workspace_bytes()  */
  CSA_ERR_CUDA = 5           /* a CUDA runtime call failed (launch, attribute, device query) */
} csa_status;

/* Bits OR-ed into *dev_status by the kernels. */
enum {
  CSA_DEV_PAGE_OOB = 1,      /* page_table entry outside [0, num_pages): page skipped      */
  CSA_DEV_RESIDENT_OOB = 2,  /* resident page id outside [0, ceil(len/64)): page skipped  */
  CSA_DEV_RANGE = 4,         /* q holds a non-finite value; or an MXFP4 input outside the exact range */
  CSA_DEV_TIMEOUT = 8,       /* an on-chip pipeline wait ran past its limit; output invalid */
  CSA_DEV_BAD_REQUEST = 16,  /* q_req entry outside [0, num_req): query treated as empty   */
  CSA_DEV_LEN_OOB = 32       /* q_len < 0, q_len > 64*pt_stride, or n_resident outside
                                [0, res_stride]: clamped                                  */
};

/*
 * Inputs of one indexer call.
 *
 * q          [num_q, num_heads, head_dim] bf16, contiguous, 16-byte aligned. The indexer
 *            query after its projection/RoPE/Hadamard chain (FlashMemory-DeepSeek-V4,
 *            "Retriever architecture"). Any finite bf16 value is accepted.
 * fused_w    [num_q, num_heads] fp32, contiguous, 4-byte aligned: weights_proj output
 *            already multiplied by head_dim^-0.5 * num_heads^-0.5.
 * kv         [num_pages] pages of 64 records, `page_stride_bytes` apart, 16-byte aligned.
 * page_table [num_req, pt_stride] int32: logical page -> physical page of each request.
 * q_req      [num_q] int32 request of each query row, or NULL for the identity map
 *            (decode: row b reads request b; then num_req must be >= num_q).
 * q_len      [num_q] int32 visible compressed records of each query row. Several rows may
 *            share one request with different bounds (chunked prefill), so the bound is
 *            per row ("DeepSeek-V4.1 native paged runtime", "Current execution scope":
 *            one scorer, each query row with its own bound and tile list).
 * resident   [num_req, res_stride] int32 logical page ids to score, or NULL to score
 *            the whole history [0, q_len). Pages of one request must be distinct.
 * n_resident [num_req] int32 entries used in each resident row (required iff resident).
 * dev_status optional int32 in device memory; kernels OR CSA_DEV_* bits into it.
 *
 * Visible records of row b (req = q_req[b], L = min(q_len[b], 64*pt_stride)):
 *   full mode      positions n in [0, L)
 *   resident mode  positions p*64 + r for each listed page p, r < 64, p*64 + r < L
 * The position n is the record's logical index in the request's history; it is what
 * top-k returns.
 *
 * Size limit: the CTAs split the rows' 256-record tiles (ceil(visible records / 256) per
 * row, counted per row even when rows share a request), plus 4 per non-empty row when
 * rows average at least 16 tiles, kept as 32-bit offsets: that total must stay below
 * 2^31 (about 5 * 10^11 records scored per call).
 */
/*
 * Record formats of the compressed-K cache (csa_index_args.record_format):
 *
 * CSA_RECORD_E4M3  132-byte records: head_dim e4m3 bytes then a little-endian fp32
 *                  scale (FlashMemory-DeepSeek-V4, "compressed_k format"); 64 records
 *                  a page, page_stride_bytes >= 8448.
 * CSA_RECORD_MXFP4 68-byte records (the published model FP4-rounds the index key and
 *                  query alike: the BatchGen #153 commit log's indexer quantisation
 *                  notes and "DeepSeek-V4.1 native paged runtime"; the pages print no
 *                  block size or layout, so the OCP MXFP4 reading is taken): 64 bytes of
 *                  e2m1 codes, element 2j in the low nibble of byte j, then the 4 UE8M0
 *                  scale bytes of the record's 32-element blocks (2^(byte - 127); 255 is
 *                  NaN). 64 records a page, page_stride_bytes >= 4352. The query is
 *                  MXFP4-rounded per head the same way (scale 2^(floor(log2 amax) - 2),
 *                  nearest e2m1 value, ties to even, saturating at 6) before the score,
 *                  which is the indexer's on the dequantised values. 64 heads only
 *                  (csa_index_score, csa_index_logits and the fused entry points; the
 *                  unfused csa_index_topk reads no keys). A record holding a NaN scale
 *                  byte is left out (CSA_DEV_RANGE). The kernel scores exactly when the
 *                  block exponents of a record, or of one query head, span at most 14;
 *                  a wider span is still scored, its smallest blocks rounded, and flagged
 *                  CSA_DEV_RANGE.
 */
#define CSA_RECORD_E4M3 0
#define CSA_RECORD_MXFP4 1

typedef struct csa_index_args {
  const void* q;
  const float* fused_w;
  int32_t num_q;
  int32_t num_heads;
  int32_t head_dim;
  int32_t reserved0;         /* must be 0 */
  const uint8_t* kv;
  int64_t num_pages;
  int64_t page_stride_bytes;
  const int32_t* page_table;
  int32_t num_req;
  int32_t pt_stride;
  const int32_t* q_req;
  const int32_t* q_len;
  const int32_t* resident;
  const int32_t* n_resident;
  int32_t res_stride;
  int32_t record_format;     /* CSA_RECORD_E4M3 (0) or CSA_RECORD_MXFP4 (1); see below */
  int32_t* dev_status;
} csa_index_args;

/* CSA_ABI_VERSION of the loaded library. */
int32_t csa_index_abi_version(void);

/* Static description of a status code; never NULL. */
const char* csa_status_str(csa_status s);

/*
 * Bytes of device workspace that csa_index_topk and csa_index_score_topk_fused need for
 * these arguments and this k. Pure host arithmetic on num_q and k (no device access):
 * 256-byte-rounded 4*(num_q+2) bytes of row offsets, then (num_q + CSA_MAX_CTAS)
 * candidate slots of 16 + 8*min(1024, k + k/2) bytes rounded up to 16, or of
 * 16 + 8*2048 bytes when num_q >= 512 (batches of that many rows take the scorer for
 * short rows, which leaves a whole row of up to 2048 candidates uncut for the merge).
 * Returns 0 when num_q < 0 or k is outside [1, CSA_MAX_K].
 */
size_t csa_index_workspace_bytes(const csa_index_args* args, int32_t k);

/*
 * Scores of every visible record ("Retriever architecture": score = sigmoid of the
 * relu'd, head-weighted sum). num_heads is 64 (the indexer) or 128 (the Level-1
 * retriever's queries; this entry point and csa_index_logits only).
 *
 * scores  [num_q, score_stride] fp32 device memory, 4-byte aligned. Row b, column c:
 *           full mode      c = logical position n, for n < L
 *           resident mode  c = j*64 + r for the j-th listed page, row r
 *         Columns of invisible records are not written.
 * score_stride >= the largest column written + 1 (full: 64*pt_stride; resident:
 *         64*res_stride is always enough).
 * Errors: CSA_ERR_INVALID_ARG (null pointers, negative sizes, score_stride too small for
 * 64*pt_stride / 64*res_stride), CSA_ERR_UNSUPPORTED, CSA_ERR_ALIGNMENT, CSA_ERR_CUDA.
 */
csa_status csa_index_score(const csa_index_args* args, float* scores, int64_t score_stride,
                           void* stream);

/*
 * csa_index_score writing the logits themselves (sum_h relu(k . q_h) * fused_w_h, before
 * the sigmoid), in the same layout, with the same arguments and errors (64 or 128 heads).
 * For callers that combine the relu'd, head-weighted sums of several scorers before the
 * sigmoid.
 */
csa_status csa_index_logits(const csa_index_args* args, float* logits, int64_t stride, void* stream);

/*
 * Top-k over a caller-provided score matrix laid out as csa_index_score writes it
 * (the "Top-k Selector" of "Two-level recall algorithm", Level 2). Only the bounds
 * fields of `args` are read: num_q, num_req, q_req, q_len, resident, n_resident,
 * res_stride, pt_stride, dev_status (q, fused_w, kv and page_table may be NULL).
 *
 * idx  [num_q, k] int32: logical positions sorted by (score desc, position asc);
 *      rows with fewer than k visible records are padded with -1.
 * vals [num_q, k] fp32: the matching scores; padding is 0.0f.
 * ws   device workspace of at least csa_index_workspace_bytes(args, k) bytes, 16-byte
 *      aligned. Contents on entry are ignored; it must not be shared by calls in flight.
 */
csa_status csa_index_topk(const float* scores, int64_t score_stride, const csa_index_args* args,
                          int32_t k, int32_t* idx, float* vals, void* ws, size_t ws_bytes,
                          void* stream);

/*
 * Exact top-k of each row from G top-k lists of that row, for context-parallel
 * scoring: one request's pages split across G GPUs, each scoring its own pages
 * ("Two-level recall algorithm", Level 2, the top-512 over the scored history)
 * and the G local lists gathered to one device. The global top-k of a row is
 * contained in the union of its local top-k lists when every k_in >= k, so the
 * merge is exact. Entries are ranked by (value desc, position asc): pass logits
 * to reproduce csa_index_score_topk_fused's order exactly, or its sigmoid
 * scores (the same order except among records whose fp32 scores tie).
 *
 * idx      [G, num_q, k_in] int32 device memory: logical positions, -1 = padding
 *          (skipped, as is a NaN value). Positions must be distinct across the G
 *          lists of a row (the shards hold disjoint pages).
 * vals     [G, num_q, k_in] fp32 device memory: each entry's logit or score.
 * out_idx  [num_q, k] int32: positions by (value desc, position asc), -1 padded.
 * out_vals [num_q, k] fp32: the matching input values unchanged (-0 becomes +0);
 *          padding 0.0f.
 * 1 <= k_in, k <= CSA_MAX_K; num_lists >= 1; any num_lists * k_in (long lists are
 * merged in rounds). No workspace.
 * Errors: CSA_ERR_INVALID_ARG (a size out of range, a null pointer with num_q > 0),
 * CSA_ERR_ALIGNMENT (pointers not 4-byte aligned), CSA_ERR_CUDA.
 */
csa_status csa_index_merge_topk(const int32_t* idx, const float* vals, int32_t num_lists, int32_t num_q,
                                int32_t k_in, int32_t k, int32_t* out_idx, float* out_vals, void* stream);

/*
 * Fused score + top-k: the scores never leave the chip ("Two-level recall algorithm",
 * Level 2, masked or full). Records are ranked by (logit desc, position asc), which is
 * the score order because sigmoid is monotone; vals hold sigmoid(logit).
 * Same idx / vals / ws contract as csa_index_topk.
 */
csa_status csa_index_score_topk_fused(const csa_index_args* args, int32_t k, int32_t* idx,
                                      float* vals, void* ws, size_t ws_bytes, void* stream);

/*
 * csa_index_score_topk_fused with one addition for profiling: `event` (a
 * cudaEvent_t passed as void*, or NULL) is recorded on `stream` between the
 * scoring kernel and the merge kernel, so a caller can time the two apart with
 * events of its own before and after the call. Same results and errors as
 * csa_index_score_topk_fused; CSA_ERR_CUDA if recording the event fails.
 */
csa_status csa_index_score_topk_fused_marked(const csa_index_args* args, int32_t k, int32_t* idx, float* vals,
                                             void* ws, size_t ws_bytes, void* stream, void* event);

/* Size of the library's built-in scratch used by csa_index_score_topk_fused_static. */
#define CSA_STATIC_SCRATCH_BYTES (4u << 20)

/*
 * Fused score + top-k that allocates nothing and needs no workspace from the
 * caller. No page describes this entry point; it exists for callers that cannot
 * hand the library device memory of their own: a plain C host without a device
 * allocator, a plugin whose host application owns every device allocation, or a
 * decode loop that must not call cudaMalloc (which may synchronise the device)
 * while it runs. It computes exactly what csa_index_score_topk_fused computes,
 * with the same argument, idx / vals and error contract, but keeps its scratch
 * (row tile offsets and per-segment candidate slots) in a CSA_STATIC_SCRATCH_BYTES
 * array that every GPU loading the library holds until the process exits.
 *
 * Limit: the call needs 256-byte-rounded 4*(num_q+2) bytes plus
 * (num_q + number of SMs) * (16 + 8*min(1024, k + k/2) rounded up to 16) bytes of
 * that array (64 rows at k = 512 on a 152-SM GB300 use about 1.3 MB); larger requests return
 * CSA_ERR_WORKSPACE before anything is launched.
 *
 * The first call on a device looks up the array's device address for that
 * device (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture, and do not use the library across a cudaDeviceReset
 * of that device (the address is kept). Every call on a device uses the same array and
 * leaves its contents behind; nothing in it has to start at zero, because each
 * call writes every byte it later reads. Calls whose kernels overlap on the GPU
 * (two streams, or two host threads) race on the array and must be serialised
 * by the caller. The library calls no cudaMalloc or cudaFree here.
 */
csa_status csa_index_score_topk_fused_static(const csa_index_args* args, int32_t k, int32_t* idx, float* vals,
                                             void* stream);

/* Ensemble of the per-layer scores in csa_recall_level1. */
enum { CSA_ENSEMBLE_MAX = 0, CSA_ENSEMBLE_MEAN = 1 };

/*
 * Level-1 recall (FlashMemory-DeepSeek-V4, "Two-level recall algorithm", Level 1, and
 * "Joint checkpoint + ensemble"): the Memory Indexer scores the full history of each query
 * row at n_layers target layers (l10, l12 and l20 on the pages) with 128-head queries
 * (the retriever's --n-heads 128); the per-layer sigmoid scores are combined per chunk,
 * by max (the pages' default, "union") or mean; a chunk is resident when the combined
 * score reaches `threshold` or it is one of the row's first `sink` or last `recent`
 * chunks ("threshold + recent + sink"). The pages print neither the threshold nor the two
 * counts: they are parameters.
 *
 * layers       host array of n_layers csa_index_args, one per layer: q [num_q, 128, 128]
 *              bf16 and fused_w [num_q, 128] of that layer's retriever, and that layer's
 *              compressed-K cache (kv, num_pages, page_stride_bytes, page_table, num_req,
 *              pt_stride). num_heads must be 128; num_q, num_req and pt_stride must be the
 *              same in every layer; the rows (q_len, q_req) are layer 0's in every layer
 *              (the other layers' q_len and q_req are not read); resident must be NULL
 *              (Level 1 reads the whole history). dev_status of layer 0 receives the
 *              device error bits of every layer.
 * ensemble     CSA_ENSEMBLE_MAX or CSA_ENSEMBLE_MEAN.
 * keep         [num_q, keep_stride] uint8 out: 1 for a resident chunk, else 0, at positions
 *              below the row's visible length (others are not written);
 *              keep_stride >= 64 * pt_stride.
 * pages        [num_q, pages_stride] int32 out: the logical pages that hold at least one
 *              resident chunk, ascending; n_pages [num_q] their count. For decode (q_req
 *              NULL) these are the Level-2 resident lists (csa_index_args.resident,
 *              n_resident with res_stride = pages_stride). pages_stride >= pt_stride.
 * scores       optional [num_q, keep_stride] fp32 out: the combined scores (written where
 *              keep is).
 * Errors: as csa_index_score for each layer, plus CSA_ERR_INVALID_ARG for n_layers outside
 * [1, 8], an unknown ensemble, a NaN threshold, negative sink or recent, strides too small,
 * layers that disagree on num_q, num_req or pt_stride, or a resident list given; and
 * CSA_ERR_WORKSPACE when ws is smaller than csa_recall_workspace_bytes; CSA_ERR_UNSUPPORTED
 * for pt_stride above 65535 * 64 pages.
 */
typedef struct csa_recall_args {
  const csa_index_args* layers;
  int32_t n_layers;
  int32_t ensemble;
  float threshold;
  int32_t sink;
  int32_t recent;
  int32_t pages_stride;
  uint8_t* keep;
  int64_t keep_stride;
  int32_t* pages;
  int32_t* n_pages;
  float* scores;
} csa_recall_args;

/* Device workspace csa_recall_level1 needs for these arguments (host arithmetic only);
 * 0 when num_q < 0 or keep_stride < 0. */
size_t csa_recall_workspace_bytes(const csa_recall_args* args);

csa_status csa_recall_level1(const csa_recall_args* args, void* ws, size_t ws_bytes, void* stream);

/* Element type of the key rows given to csa_index_write_keys. */
enum { CSA_KEYS_F32 = 0, CSA_KEYS_BF16 = 1 };

/*
 * Rows for csa_index_write_keys, the compressed-K writer: the step before the
 * indexer path that stores new keys in the cache's record format (the BatchGen
 * #153 commit log's store kernel for the "[128B fp8 | 4B fp32 scale]" layout of
 * FlashMemory-DeepSeek-V4, "compressed_k format").
 *
 * keys       [n, 128] of key_dtype (CSA_KEYS_F32 or CSA_KEYS_BF16), contiguous, 16-byte
 *            aligned.
 * row_req    [n] int32 request of each row, or NULL for row i -> request i.
 * row_pos    [n] int32 logical record position of each row in its request's history.
 * kv, num_pages, page_stride_bytes, page_table, num_req, pt_stride: the cache, as in
 *            csa_index_args; kv is written.
 * dev_status optional int32 in device memory for CSA_DEV_* bits.
 */
typedef struct csa_write_args {
  const void* keys;
  int32_t key_dtype;
  int32_t reserved0;         /* must be 0 */
  int64_t n;
  const int32_t* row_req;
  const int32_t* row_pos;
  uint8_t* kv;
  int64_t num_pages;
  int64_t page_stride_bytes;
  const int32_t* page_table;
  int32_t num_req;
  int32_t pt_stride;
  int32_t* dev_status;
} csa_write_args;

/*
 * Quantises each key row x and stores it as the record at page_table[req][pos / 64],
 * row pos % 64 of that page:
 *   amax   = max_d |x_d|
 *   scale  = amax / 448                            (binary32, round to nearest even)
 *   code_d = e4m3(x_d / scale)                     (x_d / scale in binary32; the nearest
 *            e4m3 value, ties to the even mantissa; magnitudes past 448 saturate)
 * A row whose scale is 0 (amax == 0, or amax / 448 underflows in binary32) is stored
 * as 128 zero codes and scale 0. Record bytes: the
 * 128 codes, then the scale little-endian. Only the targeted records are written;
 * rows must target distinct records (otherwise one of them wins).
 * Device errors (that row is not written; checked in this order, one bit per row):
 * request outside [0, num_req) CSA_DEV_BAD_REQUEST; position outside [0, 64*pt_stride)
 * CSA_DEV_LEN_OOB; physical page outside [0, num_pages) CSA_DEV_PAGE_OOB; a non-finite
 * value CSA_DEV_RANGE.
 * Host errors: CSA_ERR_INVALID_ARG (null pointers, n < 0, unknown key_dtype, reserved0
 * != 0, num_req or pt_stride < 1, page_stride_bytes < 64*132 or not a multiple of 16,
 * num_pages < 1), CSA_ERR_ALIGNMENT (keys, kv or row arrays misaligned), CSA_ERR_CUDA.
 * n == 0 launches nothing and returns CSA_OK.
 */
csa_status csa_index_write_keys(const csa_write_args* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA_INDEX_H */
