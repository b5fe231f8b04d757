/*
 * stof.h -- C ABI of libstof.so: masked multi-head attention (MHA) forward
 * over an arbitrary sparse mask held in STOF's two-level format, on one
 * NVIDIA GB300 (sm_103a).
 *
 * Source of the method: "Accelerating Sparse Transformer Inference on GPU"
 * (Dai et al., arXiv 2506.06095).  Passages cited below:
 *   [ABS]  arXiv abstract: STOF maps MHA to row-wise or block-wise kernels,
 *          each with its own storage format, chosen by analytical modelling.
 *   [FMT]  gist.science technical summary, Methodology 1 "Unified MHA
 *          module", two-level storage format: BSR over outer tiles (OT);
 *          empty OTs skipped globally; "full" OTs (all elements valid) and
 *          "partial" OTs (mixed) tracked by pointer arrays; every 8x8 inner
 *          tile (IT) of a partial OT is one uint64 bitmap (exact masking
 *          without materialising the sparse matrix).
 *   [ROW]  same section, dual-kernel strategy, row-wise kernel: for high
 *          sparsity and short sequences; Q sliced into rows; warp-level
 *          shuffles; no inter-warp synchronisation.
 *   [BLK]  same section, block-wise kernel: general case; Q, K, V split
 *          into sub-blocks staged in shared memory with asynchronous copies
 *          that overlap memory transfer and compute.
 *   [SEL]  same section, kernel selection: an analytical model picks the
 *          row-wise or the block-wise kernel from mask sparsity and
 *          sequence length.
 *   [PROB] same page, Problem statement: arbitrary masks (causal, sliding
 *          window, random, BigBird); work on masked entries is skipped, not
 *          computed and reset afterwards.
 *
 * Conventions of this library (the pages leave them open):
 *   - Q, K, V, O are [B][H][L][d] row-major, contiguous, fp16 or bf16,
 *     16-byte aligned device memory.  d is 32, 64, 128 or 256 (the
 *     block-wise kernels take 64 and 128).
 *   - A mask is uint8 [n_masks][L][L] (query row i, key column j); an
 *     element is valid iff its byte is non-zero.  Head (b, h) uses mask
 *     number b * mask_stride_b + h * mask_stride_h.
 *   - Scores accumulate in fp32; the softmax runs in fp32; P is rounded to
 *     the input type before P*V; O is rounded to nearest even.  A query row
 *     with no valid key gets O = 0.
 *   - All device pointers are owned by the caller.  The library allocates
 *     no device memory; the format's arrays live in a caller-provided
 *     workspace.
 *   - Every call that takes a stream is asynchronous on that stream (a
 *     cudaStream_t passed as void*; NULL is the legacy default stream).
 *     Host-side validation happens before any launch and returns an error
 *     without touching device memory.  Errors detected on the device set a
 *     device error word, reported by stof_format_sync().  The library never
 *     traps.
 */
#ifndef STOF_H_
#define STOF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define STOF_VERSION 3

typedef enum {
  STOF_OK = 0,
  STOF_ERR_INVALID_ARG = 1,  /* null pointer, negative size, unknown enum value */
  STOF_ERR_SHAPE = 2,        /* sizes inconsistent, not tile-divisible where required, or too large */
  STOF_ERR_DTYPE = 3,        /* unknown element type */
  STOF_ERR_ALIGNMENT = 4,    /* a pointer is not aligned as required */
  STOF_ERR_WORKSPACE = 5,    /* workspace smaller than stof_encode_workspace_bytes() */
  STOF_ERR_UNSUPPORTED = 6,  /* well-formed but not implemented (head dim, tile size) */
  STOF_ERR_DEVICE = 7,       /* a kernel reported an error through the device error word */
  STOF_ERR_CUDA = 8,         /* CUDA runtime error (no device, launch failure, ...) */
  STOF_ERR_NOT_SYNCED = 9    /* host tile counts needed but stof_format_sync() not called */
} stof_status;

typedef enum { STOF_F16 = 0, STOF_BF16 = 1 } stof_dtype;

typedef enum {
  STOF_KERNEL_AUTO = -1,      /* use stof_select_kernel() on the format's density */
  STOF_KERNEL_ROWWISE = 0,    /* [ROW] */
  STOF_KERNEL_BLOCKWISE = 1   /* [BLK] */
} stof_kernel;

/* Device error word bits (stof_format.device_error after a sync). */
#define STOF_DEVERR_LOOKBACK_TIMEOUT 0x1 /* encoder: a predecessor never published */
#define STOF_DEVERR_PIPE_TIMEOUT 0x2     /* block-wise kernel: a pipeline wait ran out */
#define STOF_DEVERR_BAD_FORMAT 0x4       /* an out-of-range column index was skipped */

/*
 * Two-level sparse mask format [FMT], filled by stof_encode_mask().
 *
 * Outer tiles are bm x bn; OT row r = m * n_tr + I numbers the OT rows of
 * all masks (mask-major).  Full and partial OTs each form a CSR over OT
 * rows: the tiles of row r are col_idx[row_ptr[r] .. row_ptr[r+1]), column
 * indices ascending, offsets global across masks.  Empty OTs are not
 * listed.  bitmaps[e] holds the (bm/8) x (bn/8) IT words of partial tile e
 * (row-major over ITs); bit (8*r + c) of an IT word is element (r, c) of
 * that 8x8 tile.
 *
 * All pointers are DEVICE memory inside the caller's workspace.  The host
 * counts are valid only after stof_format_sync().
 *
 * The attention kernels read the arrays as an stof_encode_* call wrote them.
 * Row pointers are trusted: a format whose row pointers were changed by the
 * caller is undefined behaviour.  Column indices are range-checked: an index
 * outside [0, n_tc) is skipped and reported as STOF_DEVERR_BAD_FORMAT.
 */
typedef struct {
  int32_t n_masks, lq, lk, bm, bn, n_tr, n_tc;
  int32_t synced;           /* 1 after a successful stof_format_sync() */
  int32_t* full_row_ptr;    /* [n_masks*n_tr + 1] */
  int32_t* full_col_idx;    /* [n_full] (capacity n_masks*n_tr*n_tc) */
  int32_t* part_row_ptr;    /* [n_masks*n_tr + 1] */
  int32_t* part_col_idx;    /* [n_part] */
  uint64_t* bitmaps;        /* [n_part][bm/8][bn/8] */
  int64_t* counts_dev;      /* [0] n_full [1] n_part [2] nnz [3] device error word */
  void* scratch;            /* encoder scratch: tile ticket and look-back state */
  int64_t n_full, n_part, nnz; /* host copies (valid when synced) */
  int64_t device_error;        /* host copy of the device error word (valid when synced) */
} stof_format;

/* Bytes of workspace stof_encode_mask() needs for these sizes, enough for
 * the worst case (every OT partial).  Returns 0 for invalid sizes. */
size_t stof_encode_workspace_bytes(int n_masks, int lq, int lk, int bm, int bn);

/*
 * Encodes a dense mask into the two-level format [FMT]: classifies every OT
 * as empty / full / partial, builds the two CSR pointer arrays by a prefix
 * sum, and packs the IT bitmaps of partial OTs, in one pass over the mask.
 *   mask       uint8 [n_masks][lq][lk], 8-byte aligned, readable by the
 *              device: device memory, or page-locked host memory mapped into
 *              the device's address space (cudaHostAlloc, or
 *              cudaHostRegister with mapping; with unified addressing the
 *              host pointer itself).  Every byte is read once, so a mask
 *              in mapped host memory is encoded at the host link's rate
 *              with no device copy of it (the format is the same).
 *   bm, bn     OT size: multiples of 8 in [8, 256].  lq and lk need not be
 *              multiples of bm and bn: a side that is not a whole number of
 *              OTs is encoded as padded to one with invalid elements, so
 *              n_tr = ceil(lq / bm), n_tc = ceil(lk / bn), and an OT that
 *              reaches past a side is partial or empty, never full.
 *   workspace  device, >= stof_encode_workspace_bytes(...) bytes, 256-byte
 *              aligned; owned by the caller and must outlive every use of fmt.
 *   fmt        host struct, overwritten; its pointers alias the workspace.
 *   stream     cudaStream_t.
 * Asynchronous.  fmt->synced is reset to 0.
 */
stof_status stof_encode_mask(const uint8_t* mask, int n_masks, int lq, int lk, int bm, int bn,
                             void* workspace, size_t ws_bytes, stof_format* fmt, void* stream);

/*
 * Same as stof_encode_mask() for a bit-packed mask: mask_bits is device
 * uint8 [n_masks][lq][lk / 8], bit c (least significant first) of byte jb
 * of row i being element (i, 8 jb + c) -- numpy's packbits along the key
 * axis with bitorder="little".  One byte of a row is then one IT row, so
 * the encoder reads an eighth of the bytes of the dense mask (in three
 * short kernels: classify, scan, fill); the format it produces is
 * identical.  The pages note that STOF keeps working at
 * sequence lengths where other systems run out of memory (scifaro.com
 * summary, Results, scalability up to 16k); a 16384-long dense mask per
 * head is 256 MB, its bit-packed form 32 MB.  Same sizes (sides that are
 * not whole OTs padded), workspace, alignment (8 bytes) and errors as
 * stof_encode_mask(); lk must be a multiple of 8 (STOF_ERR_SHAPE otherwise).
 */
stof_status stof_encode_mask_bits(const uint8_t* mask_bits, int n_masks, int lq, int lk, int bm, int bn,
                                  void* workspace, size_t ws_bytes, stof_format* fmt, void* stream);

/*
 * Same as stof_encode_mask(), for callers that cannot allocate device
 * memory at this point -- for instance code running inside a framework's
 * memory pool or allocator callback, or a pre-planned inference runtime
 * where every buffer is laid out ahead of time -- and so cannot provide
 * scratch space beyond the workspace they already own.  The paper has no
 * counterpart; this is a convenience of this library.
 *   - Allocates nothing: the encoder's scratch (its tile ticket and one
 *     look-back word per chunk) is a static device array inside
 *     libstof.so, 1 MiB + 8 bytes, held by every GPU that loads the
 *     library until the process exits.
 *   - Size limit: at most 131072 chunks, a chunk being one OT row band of
 *     W mask columns: chunks = n_masks * ceil(lq / bm) * ceil(n_tc / w)
 *     with n_tc = ceil(lk / bn) and w = min(n_tc, max(1, 1024 / bn)) OTs
 *     (W = w * bn = 1024 columns for bn = 128).
 *     Larger masks return STOF_ERR_SHAPE before any launch.  The
 *     16384 x 16384, 32-mask workload needs 65536 chunks.
 *   - The workspace (same size as for stof_encode_mask) receives the
 *     format; its scratch section is not used.
 *   - The first call on a device looks up the static array's device
 *     address (with that device current) and keeps it for the life of the
 *     process; make that first call before any stream capture.  A device
 *     reset (cudaDeviceReset) between calls is not supported: the kept
 *     address would then be stale.
 *   - All calls share the one array, which keeps the last call's contents
 *     (the call clears what must start at zero): calls that may overlap on
 *     the GPU, from several streams or threads, race and must not be made.
 */
stof_status stof_encode_mask_noalloc(const uint8_t* mask, int n_masks, int lq, int lk, int bm, int bn,
                                     void* workspace, size_t ws_bytes, stof_format* fmt, void* stream);

/*
 * A mask given by a rule instead of stored elements: the union of the
 * pattern families the pages name -- a diagonal band (causal, sliding
 * window), global tokens (Longformer) and a block pattern (BigBird)
 * [PROB]; gist.science technical summary, Experimental results.  Element
 * (i, j) of a mask is valid iff
 *     band_lo <= i - j <= band_hi             (empty band if band_lo > band_hi)
 *  or bit i of global_rows is set              (query row i sees every key)
 *  or bit j of global_cols is set              (every query row sees key j)
 *  or bit (i / block) * (lk / block) + j / block of blocks is set.
 * A bitset is DEVICE memory: uint32 words, bit b at position b % 32 of
 * word b / 32 (least significant first), 4-byte aligned; NULL is empty.
 *   global_rows   ceil(lq / 32) words;   global_cols   ceil(lk / 32) words;
 *   blocks        ceil((lq / block) * (lk / block) / 32) words;
 *   block         edge of a block: a multiple of 8 dividing lq and lk
 *                 (read only when blocks is not NULL).
 * Examples: causal = {0, INT32_MAX}; causal sliding window w = {0, w - 1};
 * symmetric window |i - j| <= w = {-w, w}.
 */
typedef struct {
  int32_t band_lo, band_hi;
  const uint32_t* global_rows;
  const uint32_t* global_cols;
  const uint32_t* blocks;
  int32_t block;
} stof_mask_rule;

#define STOF_MAX_RULES 64

/*
 * Encodes n_masks parametric masks (rules: HOST array of n_masks rules, at
 * most STOF_MAX_RULES) into the two-level format [FMT].  The result is the
 * format that stof_encode_mask() gives for the dense masks the rules define,
 * but no mask is read: the encoder computes every IT word from the rule, so
 * long sequences need no L x L mask in memory at all (the pages' long-
 * sequence results: scifaro.com summary, Results).  The rules are copied at
 * the call; the bitsets they point to must stay valid until the encoding is
 * done on the stream.  Sizes, workspace and errors as stof_encode_mask();
 * STOF_ERR_UNSUPPORTED for more than STOF_MAX_RULES masks, STOF_ERR_SHAPE
 * for a bad block edge, STOF_ERR_ALIGNMENT for a bitset not 4-byte aligned.
 */
stof_status stof_encode_rules(const stof_mask_rule* rules, int n_masks, int lq, int lk, int bm, int bn,
                              void* workspace, size_t ws_bytes, stof_format* fmt, void* stream);

/* Blocks until the work queued on stream is done, copies the tile counts
 * and the device error word into fmt, and sets fmt->synced.  Returns
 * STOF_ERR_DEVICE if the device error word is non-zero. */
stof_status stof_format_sync(stof_format* fmt, void* stream);

/* Analytic kernel choice [SEL]: row-wise or block-wise from the mask
 * density (valid elements / all elements, in [0, 1]), the sequence length
 * and the head dimension, for one head whose mask lists every OT (the
 * worst case of an arbitrary mask).  The model compares each kernel's
 * predicted time, linear in its work: the row-wise kernel's in query rows
 * and valid (query, key) pairs, the block-wise kernel's in listed OTs and
 * query tiles (coefficients fitted to both kernels' GB300 times).  Pure host
 * arithmetic and deterministic; invalid arguments give
 * STOF_KERNEL_BLOCKWISE.  Same as stof_select_kernel_heads(density,
 * seq_len, head_dim, 1, -1). */
stof_kernel stof_select_kernel(double density, int seq_len, int head_dim);

/* The same model for `heads` heads (B * H) of one call, whose masks list
 * tiles_per_row 128x128 OTs per 128-row query tile on average (a negative
 * value: every OT).  The row-wise kernel's fixed cost per query row is a few
 * dependent memory round trips, so it wins only while the whole call is
 * small and sparse; stof_mha_fwd(STOF_KERNEL_AUTO) uses this with the call's
 * B * H and the format's tile counts. */
stof_kernel stof_select_kernel_heads(double density, int seq_len, int head_dim, int64_t heads, double tiles_per_row);

/*
 * Masked MHA forward [ABS][PROB]:
 *   O[b,h,i,:] = sum_{j valid} softmax_j(scale * Q[b,h,i,:].K[b,h,j,:]) V[b,h,j,:]
 * over the valid keys of query row i in mask b*mask_stride_b + h*mask_stride_h;
 * rows without valid keys give 0.  Only listed OTs are touched; full OTs
 * need no mask test, partial OTs are masked through their IT bitmaps.
 *   q, k, v, o  device [B][H][L][d], dt, 16-byte aligned; o is written.
 *   L           == fmt->lq == fmt->lk, any length (a last OT row and column
 *               that reach past L are padded: rows past L are computed and
 *               not stored, keys past L are never valid).
 *   d           32, 64, 128 or 256; the block-wise kernel takes 64 and 128
 *               (STOF_ERR_UNSUPPORTED if forced on another), AUTO runs the
 *               row-wise kernel for 32 and 256 (at most 2 query rows per
 *               warp at d = 256).
 *   scale       any finite value; the softmax is taken over scale * Q.K
 *               (a negative scale favours the smallest dot products, a zero
 *               scale averages the valid V rows).
 *   fmt         an encoded format (stof_encode_mask) for masks of size L.
 *   which       STOF_KERNEL_ROWWISE [ROW], STOF_KERNEL_BLOCKWISE [BLK]
 *               (needs bm == 128 and bn == 64 or 128; else
 *               STOF_ERR_UNSUPPORTED) or STOF_KERNEL_AUTO (needs a synced
 *               fmt): the fastest measured candidate that stof_tune()
 *               cached for (L, d, the density's bucket) among those on the
 *               format's OT width, if there is one; else the analytic model
 *               [SEL] (stof_select_kernel_heads with B * H and the format's
 *               tiles), falling back to row-wise for tile sizes the
 *               block-wise kernel does not take.  stof_mha_plan() tells
 *               which.
 * Asynchronous on stream.  For d = 64 the block-wise kernel may run
 * persistent CTAs that take query tiles from a work counter kept in two
 * words of the format's workspace (zeroed by every encoder, and zeroed
 * again by the kernel's last CTA when it ends): calls that use the same
 * format must not overlap on the GPU (one stream, or streams ordered by
 * events); calls with different formats may.
 */
stof_status stof_mha_fwd(const void* q, const void* k, const void* v, stof_dtype dt, int B, int H,
                         int L, int d, float scale, const stof_format* fmt,
                         int64_t mask_stride_b, int64_t mask_stride_h, stof_kernel which, void* o,
                         void* stream);

/*
 * stof_mha_fwd() with Lq query rows and Lk keys per head (attention of one
 * sequence over another, e.g. a decoder over an encoder's output):
 *   q, o      device [B][H][Lq][d];  k, v  device [B][H][Lk][d].
 *   fmt       encodes masks of Lq rows and Lk columns (fmt->lq == Lq,
 *             fmt->lk == Lk); the masks, kernels and errors are those of
 *             stof_mha_fwd(), which is this call with Lq = Lk = L.  AUTO
 *             uses a stof_tune() result only when Lq == Lk.
 */
stof_status stof_mha_fwd_cross(const void* q, const void* k, const void* v, stof_dtype dt, int B, int H, int Lq,
                               int Lk, int d, float scale, const stof_format* fmt, int64_t mask_stride_b,
                               int64_t mask_stride_h, stof_kernel which, void* o, void* stream);

/* Where a plan's choice came from. */
#define STOF_PLAN_FORCED 0    /* the caller named the kernel */
#define STOF_PLAN_ANALYTIC 1  /* stof_select_kernel() on the format's density [SEL] */
#define STOF_PLAN_TUNED 2     /* a cached stof_tune() measurement */

/* What one stof_mha_fwd() call runs. */
typedef struct {
  stof_kernel kernel;  /* STOF_KERNEL_ROWWISE or STOF_KERNEL_BLOCKWISE */
  int stages;          /* block-wise K/V ring depth; 0 for the row-wise kernel */
  int persistent;      /* block-wise: 1 = persistent CTAs (d = 64), 0 = one CTA per query tile */
  int source;          /* STOF_PLAN_FORCED, STOF_PLAN_ANALYTIC or STOF_PLAN_TUNED */
  int rows_per_warp;   /* row-wise: query rows per warp (1, 2 or 4); 0 for the block-wise kernel */
  int exp_split;       /* block-wise: 1 = one key pair in eight takes its exponentials on the FMA pipe
                          (a Remez-fitted polynomial) instead of the special-function unit; else 0 */
  int softmax_warpgroups; /* block-wise softmax warpgroups: 2, or 4 (persistent, d = 64); 0 row-wise */
} stof_plan;

/*
 * The plan stof_mha_fwd(q, k, v, dt, B, H, L, d, scale, fmt, ..., which, ...)
 * follows, without running it: fills *out and returns STOF_OK, or the
 * status that call would return for these sizes, format and `which`.
 * Pure host code.
 */
stof_status stof_mha_plan(const stof_format* fmt, int B, int H, int L, int d, stof_kernel which, stof_plan* out);

/*
 * stof_mha_fwd() run exactly as *plan says: its kernel, and for the
 * block-wise kernel its ring depth, variant, exp split and softmax
 * warpgroup count (plan->source is ignored).  Arguments, layout and errors
 * as stof_mha_fwd(); STOF_ERR_UNSUPPORTED for a setting these sizes do not
 * admit, STOF_ERR_INVALID_ARG for exp_split other than 0 or 1 or a ring
 * depth outside 0..8.  Admitted: row-wise on any OT size with 1, 2 or 4
 * query rows per warp (0: the library's choice) and exp_split and
 * softmax_warpgroups 0; block-wise on 128x128 OTs one CTA per query tile
 * with ring depth 2 or 3 (d = 128) or 2, 3 or 4 (d = 64), persistent CTAs
 * with ring depth 2, 3 or 4 (d = 64 only); on 128x64 OTs the default depth
 * (3 per query tile, 4 persistent); the exp split on 128x128 OTs at the
 * default depth (3 per query tile, 4 persistent); four softmax warpgroups
 * on 128x128 OTs, persistent, ring depth 4, d = 64, without the exp split
 * (softmax_warpgroups 0 means 2).  A plan from stof_mha_plan() or a
 * stof_tune_result's candidate is always admitted for the sizes it was
 * made for.
 */
stof_status stof_mha_fwd_plan(const void* q, const void* k, const void* v, stof_dtype dt, int B, int H, int L, int d,
                              float scale, const stof_format* fmt, int64_t mask_stride_b, int64_t mask_stride_h,
                              const stof_plan* plan, void* o, void* stream);

/*
 * Measured parameter choice for the MHA step, with a result cache.  The
 * pages' tuner samples kernel parameters (block size, pipeline stages) by
 * running them once the operator boundaries are fixed, and caches what it
 * measured (gist.science technical summary, Methodology 2, two-stage
 * tuning, stage 2 "parameter sampling"; the cache: same page, the lay
 * summary's "autopilot" that remembers what worked).  The candidates:
 *   0-2    row-wise kernel, 128x128 OTs, 1, 2, 4 query rows per warp;
 *   3-5    block-wise, 128x128 OTs, one CTA per query tile, K/V ring depth
 *          3, 2, 4 (depth 4 at d = 64 only: shared memory);
 *   6-8    block-wise, 128x128 OTs, persistent CTAs (d = 64 only), ring
 *          depth 4, 3, 2;
 *   9      block-wise, 128x64 OTs, default variant and ring depth;
 *   10     block-wise, 128x128 OTs, one CTA per query tile, ring depth 3,
 *          exp split;
 *   11     block-wise, 128x128 OTs, persistent (d = 64 only), ring depth 4,
 *          exp split;
 *   12     block-wise, 128x128 OTs, persistent (d = 64 only), ring depth 4,
 *          four softmax warpgroups.
 */
#define STOF_TUNE_CANDIDATES 13
typedef struct {
  stof_kernel kernel;        /* fastest candidate */
  int bn;                    /* its OT width (bm = 128) */
  float ms;                  /* its time per stof_mha_fwd call */
  double density;            /* density of the tuned mask */
  int stages;                /* its K/V ring depth (0 for row-wise) */
  int persistent;            /* 1 if it runs persistent CTAs */
  int rows_per_warp;         /* row-wise: its query rows per warp (0 for block-wise) */
  int exp_split;             /* block-wise: 1 if its exp split is on */
  int softmax_warpgroups;    /* block-wise: its softmax warpgroups (2 or 4; 0 row-wise) */
  stof_kernel cand_kernel[STOF_TUNE_CANDIDATES];
  int cand_bn[STOF_TUNE_CANDIDATES];
  int cand_stages[STOF_TUNE_CANDIDATES];        /* ring depth the candidate ran with (0 row-wise) */
  int cand_persistent[STOF_TUNE_CANDIDATES];    /* 1 persistent, 0 one CTA per query tile */
  int cand_rows_per_warp[STOF_TUNE_CANDIDATES]; /* row-wise rows per warp (0 block-wise) */
  int cand_exp_split[STOF_TUNE_CANDIDATES];     /* 1 exp split on */
  int cand_softmax_warpgroups[STOF_TUNE_CANDIDATES]; /* block-wise softmax warpgroups (0 row-wise) */
  float cand_ms[STOF_TUNE_CANDIDATES];          /* -1 for a candidate the sizes do not admit */
} stof_tune_result;

/* Workspace bytes stof_tune() needs (the largest encode workspace over the
 * candidates' OT sizes); 0 for invalid sizes. */
size_t stof_tune_workspace_bytes(int n_masks, int L);

/*
 * Encodes the mask for each candidate OT size, runs every candidate kernel
 * (one untimed call, then three timed with CUDA events) and returns the
 * fastest in *out; the result is also cached under (L, d, density bucket),
 * where stof_mha_fwd(STOF_KERNEL_AUTO) finds it.
 * Arguments as for stof_encode_mask() and stof_mha_fwd(); the workspace must
 * hold stof_tune_workspace_bytes(n_masks, L) bytes and o is overwritten.
 * Blocks until the timing is done.  A candidate whose run reports a device
 * error ends the call with that error.
 */
stof_status stof_tune(const uint8_t* mask, int n_masks, const void* q, const void* k, const void* v,
                      stof_dtype dt, int B, int H, int L, int d, float scale, int64_t mask_stride_b,
                      int64_t mask_stride_h, void* workspace, size_t ws_bytes, void* o, stof_tune_result* out,
                      void* stream);

/* Cached result for (L, d, the density's bucket): 1 and *out filled (when
 * out is not NULL) if present, else 0.  Thread-safe; the cache lives for the
 * process. */
int stof_tune_lookup(int L, int d, double density, stof_tune_result* out);

/* Empties the cache. */
void stof_tune_clear(void);

/* The cache's density bucket: round(2 log2(density)), clamped to >= -60;
 * -61 for density 0. */
int stof_tune_density_bucket(double density);

/*
 * Output projection after the MHA with a fused epilogue (gist.science
 * technical summary, Methodology 2: fusion carried past the MHA layer into
 * the operators that follow it):
 *   y[b, l, n] = sum_{h, c} O[b, h, l, c] * W[n, h*d + c] + bias[n] + residual[b, l, n]
 *   o         device [B][H][L][d] (the MHA output), dt.
 *   w         device [N][H*d] row-major (a linear layer's weight), dt.
 *   bias      device [N] or NULL; residual device [B][L][N] or NULL; dt.
 *   y         device [B][L][N], written; must not overlap the inputs.
 *   device_error  device int64 word that a pipeline timeout ORs
 *             STOF_DEVERR_PIPE_TIMEOUT into, or NULL.
 * fp32 accumulation; bias and residual are added in fp32 and y is rounded
 * once to nearest even.  Requires d = 64 or 128, N % 256 == 0 and 16-byte
 * aligned pointers; any L.  Asynchronous on stream.
 */
stof_status stof_oproj_fwd(const void* o, const void* w, const void* bias, const void* residual,
                           stof_dtype dt, int B, int H, int L, int d, int N, void* y,
                           int64_t* device_error, void* stream);

/*
 * stof_oproj_fwd() followed by a LayerNorm over the N output features of
 * each token -- the operator that closes a post-norm transformer sublayer,
 * fused the same way (gist.science technical summary, Methodology 2):
 *   z = concat_heads(O) W^T + bias + residual
 *   y[b, l, :] = (z - mean) / sqrt(var + eps) * gamma + beta
 * with mean and var (population variance) of z[b, l, :] as rounded to dt.
 * The GEMM's epilogue writes z and each (token, 256-feature tile)'s mean and
 * sum of squared deviations to `workspace`; a second pass merges them and
 * normalises y in place.
 *   gamma, beta  device [N] or NULL (1 and 0), dt, 16-byte aligned.
 *   eps          > 0, finite.
 *   workspace    device, >= stof_oproj_ln_workspace_bytes(B, L, N) bytes,
 *                16-byte aligned; caller-owned scratch.
 * Other arguments, requirements and errors as stof_oproj_fwd().
 * Asynchronous on stream.
 */
stof_status stof_oproj_ln_fwd(const void* o, const void* w, const void* bias, const void* residual, const void* gamma,
                              const void* beta, float eps, stof_dtype dt, int B, int H, int L, int d, int N, void* y,
                              void* workspace, size_t ws_bytes, int64_t* device_error, void* stream);

/* Workspace bytes of stof_oproj_ln_fwd(): 8 per (token, 256-feature tile);
 * 0 for invalid sizes. */
size_t stof_oproj_ln_workspace_bytes(int B, int L, int N);

/*
 * Diagnostic of the failure handling (the paper has no counterpart): every
 * pipeline wait in this library's kernels is bounded in wall time and, when
 * it runs out, ORs an error bit into a device error word and lets the
 * kernel finish instead of hanging.  This call launches one CTA that waits,
 * through that same bounded wait, on a barrier nothing ever arrives on; after
 * `seconds` (in (0, 10]) it ORs STOF_DEVERR_PIPE_TIMEOUT into *device_error
 * (device int64, 8-byte aligned) and exits.  Asynchronous on stream.
 */
stof_status stof_check_bounded_wait(int64_t* device_error, double seconds, void* stream);

/*
 * The block-wise kernels' FMA-pipe exp2 (the exp split's polynomial) on n
 * inputs: y[i] = 2^x[i] computed as 2^rint(x) * p(x - rint(x)) with a
 * degree-4 polynomial p (p(0) = 1; relative error at most 2.9e-6 on
 * [-1/2, 1/2]); 0 for x < -125 and at -inf.  For x <= 127.  x and y are
 * device fp32 arrays (4-byte aligned, may be the same array).  Lets a test
 * check the polynomial against exp2.  STOF_ERR_INVALID_ARG for n < 0 or a
 * NULL array with n > 0.  Asynchronous on stream.
 */
stof_status stof_ex2_fma(const float* x, float* y, int64_t n, void* stream);

/* Static description of a status code. */
const char* stof_status_string(stof_status s);

/* STOF_VERSION of the built library. */
int stof_version(void);

/* Text of the last CUDA runtime error this library saw on the calling
 * thread ("no error" if none), to explain a STOF_ERR_CUDA status. */
const char* stof_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* STOF_H_ */
