/*
 * msa.h -- C ABI of the MiniMax Sparse Attention (MSA) layer hot path on one
 * GB300 (sm_103a).
 *
 * MSA runs in two stages.  An Index Branch scores every Bk-token KV block for
 * each query and KV (GQA) group and keeps k blocks; exact softmax attention
 * then runs against only those blocks, in causal prefill and in paged decode.
 * Sources, by page title and passage:
 *   [serving]  "MiniMax M3 preparado para inferencia en produccion" (community
 *              post on the M3 serving report), paragraphs "KV-Block-Major",
 *              "MSA con paged attention" and "MSA opera en dos etapas".
 *   [agents]   "MiniMax M3: Como la atencion dispersa hace practicos a los
 *              agentes de largo alcance", MSA paragraph, its figure caption and
 *              the bullet "Costo predecible a cualquier longitud" (Bk = 128,
 *              k = 16: 2048 tokens per query and GQA group).
 *   [M2]       article on the MiniMax M2 report, section "MiniMax Sparse
 *              Attention (MSA) y escalado subcuadratico entrante" (block
 *              selection on real, uncompressed KV over a GQA backbone).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless a
 *    comment says otherwise.  The library never allocates device memory, never
 *    synchronises the device or a stream, and keeps no state between calls
 *    except a per-device cache of kernel attributes.
 *  - Work is enqueued on `stream` and runs asynchronously.  A call that returns
 *    MSA_OK has enqueued all of its work; results are ready when the stream is.
 *  - Arguments are validated on the host first.  On any error nothing is
 *    enqueued and msa_last_error_string() (thread-local) says why.
 *  - bf16 tensors are raw 16-bit bfloat16 storage (`void*`); accumulation is
 *    fp32.  Strides are given in ELEMENTS for every dimension except the
 *    innermost, which is always contiguous.  Strides of tensors that the
 *    kernels stage with TMA must be multiples of 16 bytes and their base
 *    pointers 16-byte aligned; bf16 vectors read with 16-byte loads likewise.
 *  - `dev_err` (optional, may be NULL) is a caller-owned device int32.  Kernels
 *    OR MSA_DEVERR_* bits into it when a device-side check fails (a bounded
 *    wait that ran out, a page id or block index outside its range); they then
 *    skip the offending work and return without trapping.  The caller clears
 *    it and reads it back when convenient.
 *  - Supported shapes: D = 128, dI = 64, Bk = 128, 1 <= HI <= 4,
 *    1 <= k <= 64, GQA ratio G = Hq / Hkv in 1..8 (Hq a multiple of Hkv).
 *    Anything else returns MSA_ERR_UNSUPPORTED.
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers */
typedef struct CUstream_st *msa_stream_t;

typedef enum msa_status {
    MSA_OK = 0,
    MSA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad stride, ... */
    MSA_ERR_UNSUPPORTED = 2,   /* a shape outside the supported set above */
    MSA_ERR_CUDA = 3,          /* a CUDA runtime call failed */
    MSA_ERR_DEVICE_CHECK = 4,  /* reserved for callers that read dev_err back */
    MSA_ERR_WORKSPACE = 5      /* workspace pointer or size too small */
} msa_status;

/* bits OR-ed into *dev_err by the kernels */
#define MSA_DEVERR_TIMEOUT 0x1   /* a bounded barrier wait ran out */
#define MSA_DEVERR_BAD_PAGE 0x2  /* a page id outside [0, num_pages) */
#define MSA_DEVERR_BAD_SEL 0x4   /* a selected block outside the causal range */
#define MSA_DEVERR_BAD_LEN 0x8   /* seq_len[b] (or a chunk's q_pos[b]) outside the pages or past nb_stride */

/* PREFILL: a causal prefill over contiguous K/V/k_idx tensors.
 * DECODE:  one query per sequence over a paged cache.
 * CHUNK:   a chunk of S queries per sequence over a paged cache: query s of
 *          sequence b sits at absolute position q_pos[b] + s and sees every
 *          cached token t <= q_pos[b] + s.  This is chunked prefill over a
 *          cached prefix, and with a small S, decode of several tokens per
 *          sequence (speculative or multi-token verification).  The chunk's
 *          own tokens must already be in the pages (msa_cache_append). */
typedef enum msa_mode {
    MSA_MODE_PREFILL = 0,
    MSA_MODE_DECODE = 1,
    MSA_MODE_CHUNK = 2
} msa_mode;

/* Library version: major * 10000 + minor * 100 + patch. */
int msa_version(void);

/* Human-readable text of the last host-side error of this thread. */
const char *msa_last_error_string(void);

/* Name of a status code. */
const char *msa_status_string(msa_status s);

/* --------------------------------------------------------------------------
 * a1. Index score
 *
 * Block relevance scores of the Index Branch ([agents], MSA paragraph and
 * caption).  The pages never print the formula; this library computes
 *     s_t = sum_{h < HI} w_h * ReLU(q_idx_h . k_idx_t)        (fp32 accumulate)
 *     c_j = max over the Bk tokens t of block j of s_t
 * for every block j strictly before the query's own block, and writes -inf for
 * the own block and every later entry up to nb_stride.  The own block is always
 * kept by selection and is never scored.
 *
 * PREFILL: query i of sequence b has own block i / Bk and scores blocks of the
 *   same sequence's index keys.
 *     q_idx [B, S, Hkv, HI, dI] bf16, strides q_idx_stride = (b, s, g, h)
 *     w     [B, S, Hkv, HI]     fp32, strides w_stride     = (b, s, g)
 *     k_idx [B, S, Hkv, dI]     bf16, strides k_idx_stride = (b, s, g); a group
 *           stride of 0 means one index-key tensor shared by all KV groups
 *     C     [B, S, Hkv, nb_stride] fp32, strides C_stride = (b, s, g),
 *           nb_stride >= ceil(S / Bk)
 * DECODE: one query per sequence at position L_b - 1 (its own token already in
 *   the cache); its own block is (L_b - 1) / Bk.  Index keys live in pages of
 *   Bk tokens: logical block j of sequence b is page seq_pt[b][j].
 *     q_idx [B, Hkv, HI, dI] bf16, strides (b, g, h, unused)
 *     w     [B, Hkv, HI]     fp32, strides (b, g, unused)
 *     k_idx page pool [num_pages, Hkv, Bk, dI] bf16, strides (page, g, t); a
 *           group stride of 0 means one pool shared by all KV groups (scored
 *           once per block for every group; HI = 4 and Hkv <= 8)
 *     seq_pt [B, max_pages] int32 (row stride max_pages), seq_len [B] int32
 *     C     [B, Hkv, nb_stride] fp32, strides (b, g, unused);
 *           nb_stride >= max over b of ceil(L_b / Bk) (entries past the own
 *           block, up to nb_stride, are written -inf).
 *   Page ids outside [0, num_pages) are not read: the block gets -inf and
 *   MSA_DEVERR_BAD_PAGE is raised.  A sequence whose length is outside
 *   [1, max_pages * Bk], or whose own block is not below nb_stride, is not
 *   scored (its row stays -inf) and raises MSA_DEVERR_BAD_LEN.
 * CHUNK: queries as in PREFILL (q_idx, w and C with the same shapes and
 *   strides, S = queries per sequence); index keys in pages as in DECODE
 *   (k_idx page pool, num_pages, seq_pt, max_pages; group stride 0 allowed).
 *   (With S <= 8, HI <= 4 and per-group keys the scores are computed by the
 *   decode kernel, all of a sequence's tokens per page read; the results are
 *   the same.)
 *   q_pos [B] int32: absolute position of query 0 of sequence b.  Query s has
 *   own block (q_pos[b] + s) / Bk and scores the blocks before it;
 *   max over b of ceil((q_pos[b] + S) / Bk) <= nb_stride <= max_pages (a
 *   larger nb_stride is rejected on the host).  A sequence with q_pos[b] < 0
 *   or whose last query's own block (q_pos[b] + S - 1) / Bk is not below
 *   nb_stride is not scored (its rows are -inf) and raises
 *   MSA_DEVERR_BAD_LEN; msa_topk_blocks with the same nb_stride rejects the
 *   same sequences.  A page id outside [0, num_pages) is not read: that
 *   block's scores are -inf in every row and MSA_DEVERR_BAD_PAGE is raised.
 * DECODE, fused selection (optional): when `sel` is non-NULL the same kernel
 *   also performs a2 (exactly what msa_topk_blocks computes with this k) on
 *   each (b, g) row as soon as the row's scores are complete, and when `pt` is
 *   also non-NULL a3 (exactly what msa_build_page_table computes).  This saves
 *   two launches per decode step.  With one index-key pool for all groups
 *   (group stride 0) and nb_stride > 2048 the call instead launches the
 *   top-k and page-table kernels after the scores (a sequence's group rows
 *   would otherwise all be selected by one CTA); the outputs are the same.  `row_scratch` is then required: B*Hkv int32
 *   of caller scratch (one completion counter per row).  Outputs are those of
 *   a2 / a3: sel [B,Hkv,k], count [B,Hkv], pt [B*Hkv,k], n and last_len [B*Hkv].
 *   scratch_zeroed = 0: the call clears row_scratch first (one memset on the
 *   stream).  scratch_zeroed = 1: the caller guarantees row_scratch is zero
 *   (freshly zero-filled, or left by a previous call) and the memset is
 *   skipped.  Either way a call that raises no device error leaves row_scratch
 *   zero; after one that does, zero it again (or pass 0).
 * ------------------------------------------------------------------------ */
typedef struct msa_index_args {
    msa_mode mode;
    int B, S, Hkv, HI, dI, Bk;
    const void *q_idx;
    int64_t q_idx_stride[4];
    const float *w;
    int64_t w_stride[3];
    const void *k_idx;
    int64_t k_idx_stride[3];
    int64_t num_pages;            /* decode */
    const int32_t *seq_pt;        /* decode */
    int64_t max_pages;            /* decode */
    const int32_t *seq_len;       /* decode */
    float *C;
    int64_t C_stride[3];
    int nb_stride;
    int32_t *dev_err;
    /* decode, optional fused a2/a3 outputs (NULL = scores only) */
    int k;
    int32_t *sel;
    int32_t *count;
    int32_t *pt;
    int32_t *n;
    int32_t *last_len;
    int32_t *row_scratch;
    int scratch_zeroed;
    const int32_t *q_pos;         /* chunk */
} msa_index_args;

msa_status msa_index_score(const msa_index_args *args, msa_stream_t stream);

/* --------------------------------------------------------------------------
 * a2. Top-k block selection
 *
 * Per (query, KV group) row keep the own block and the k-1 best earlier blocks,
 * ordered by (score descending, block index ascending); when the row has at
 * most k-1 earlier blocks keep them all ([agents], "Costo predecible": k
 * blocks including the query's own).  Output is ascending and padded with -1;
 * the own block, the largest selected index, comes last.
 *   PREFILL rows (b, s, g): own block s / Bk.   C strides (b, s, g).
 *     sel [B, S, Hkv, k] int32, count [B, S, Hkv] int32 (dense).
 *   DECODE rows (b, g): own block (seq_len[b] - 1) / Bk.  C strides (b, g, -).
 *     sel [B, Hkv, k] int32, count [B, Hkv] int32 (dense).
 *   CHUNK rows (b, s, g): own block (q_pos[b] + s) / Bk; C, sel and count as
 *     in PREFILL.  A sequence with q_pos[b] < 0, or whose last query's own
 *     block (q_pos[b] + S - 1) / Bk is not below nb_stride, gets count 0 and
 *     all -1 selections in every row, and MSA_DEVERR_BAD_LEN.
 * Scores are compared as fp32 (-0 equals +0); NaN scores rank below -inf.
 * A decode row whose length is outside [1, nb_stride * Bk] gets count 0, an
 * all -1 selection and MSA_DEVERR_BAD_LEN.
 * ------------------------------------------------------------------------ */
typedef struct msa_topk_args {
    msa_mode mode;
    int B, S, Hkv, Bk, k;
    const float *C;
    int64_t C_stride[3];
    int nb_stride;                /* entries per score row (as given to msa_index_score) */
    const int32_t *seq_len;       /* decode */
    int32_t *sel;
    int32_t *count;
    int32_t *dev_err;
    const int32_t *q_pos;         /* chunk */
} msa_topk_args;

msa_status msa_topk_blocks(const msa_topk_args *args, msa_stream_t stream);

/* --------------------------------------------------------------------------
 * a3. Decode page table from the selected blocks
 *
 * The KV-group dimension is flattened into the batch so that a fixed-page
 * attention kernel can serve per-group selections ([serving], "MSA con paged
 * attention").  Row r = b * Hkv + g:
 *     pt[r][s]    = seq_pt[b][sel[b][g][s]]  for s < count[b][g], else -1
 *     n[r]        = count[b][g]
 *     last_len[r] = valid tokens of the row's last selected page (its own
 *                   block): seq_len[b] - Bk * ((seq_len[b] - 1) / Bk).
 * sel [B, Hkv, k], count [B, Hkv], seq_pt [B, max_pages], seq_len [B];
 * pt [B*Hkv, k], n [B*Hkv], last_len [B*Hkv] (all int32, dense).
 * A selected index outside [0, own block] yields page -1 and MSA_DEVERR_BAD_SEL.
 * ------------------------------------------------------------------------ */
msa_status msa_build_page_table(const int32_t *sel, const int32_t *count,
                                const int32_t *seq_pt, int64_t max_pages,
                                const int32_t *seq_len, int B, int Hkv, int k, int Bk,
                                int32_t *pt, int32_t *n, int32_t *last_len,
                                int32_t *dev_err, msa_stream_t stream);

/* --------------------------------------------------------------------------
 * a3'-a4-a6. Sparse attention, causal prefill (KV-block-major)
 *
 * For every query i, q-head hq (KV group g = hq / G) and selected block j of
 * (i, g): exact softmax attention over the tokens t of the selected blocks with
 * t <= i ([M2]).  The kernel iterates over KV blocks in the outer loop: it
 * inverts the selection into per-(b, g, j) query lists, stages each selected
 * block's K and V once in shared memory, runs every query that chose it
 * against it, and combines the per-block partials with a log-sum-exp merge
 * ([serving], "KV-Block-Major").
 *     Q [B, S, Hq, D] bf16 strides (b, s, h); K, V [B, S, Hkv, D] bf16 strides
 *     (b, s, g); sel [B, S, Hkv, k] and count [B, S, Hkv] int32 (dense, as
 *     written by msa_topk_blocks);
 *     O [B, S, Hq, D] bf16 (dense), LSE [B, S, Hq] fp32 (dense, natural log,
 *     softmax_scale included).
 * A selected block outside [0, own block] is ignored and raises
 * MSA_DEVERR_BAD_SEL.
 * mode = MSA_MODE_CHUNK (mode 0 = PREFILL; DECODE is not accepted here): the
 *   queries are a chunk at absolute positions q_pos[b] + s (q_pos [B] int32)
 *   and K, V are page pools [num_pages, Hkv, Bk, D] bf16 with strides K_stride
 *   = V_stride = (page, g, t); logical block j of sequence b is page
 *   seq_pt[b * max_pages + j].  Query s sees the tokens t <= q_pos[b] + s of
 *   its selected blocks.  A selected block at or past max_pages raises
 *   MSA_DEVERR_BAD_SEL and a page id outside [0, num_pages) raises
 *   MSA_DEVERR_BAD_PAGE; either slot is ignored.  Pool slots past a sequence's
 *   last token must hold finite values (a zero-filled pool does): their
 *   probabilities are 0, and 0 times a NaN or an infinity is NaN.
 *   With S <= 8 queries per sequence (a few decode tokens, e.g. draft
 *   verification), Q dense over (b, s) (Q_stride[0] = S * Q_stride[1]) and K,
 *   V with equal strides, the rows (b, s, g) run as a decode batch of B * S
 *   sequences through the paged decode attention (a page table of each row's
 *   selected pages, then one attention launch with the merge fused); the
 *   workspace then holds that path's page table and partials and does not
 *   depend on chunk_queries.
 * Workspace: caller-owned device scratch of ws_bytes.  Queries are processed in
 * chunks sized to fit; msa_sparse_attn_prefill_workspace_size(args, q) gives
 * the bytes needed for chunks of q queries (q >= 1; in CHUNK mode it reads
 * mode, max_pages and the Q, K and V strides too); larger workspaces mean
 * fewer passes.  The workspace must stay untouched until the stream has run
 * the call.  softmax_scale <= 0 selects 1 / sqrt(D).
 * ------------------------------------------------------------------------ */
typedef struct msa_prefill_args {
    int B, S, Hq, Hkv, D, Bk, k;
    float softmax_scale;
    const void *Q;
    int64_t Q_stride[3];
    const void *K;
    int64_t K_stride[3];
    const void *V;
    int64_t V_stride[3];
    const int32_t *sel;
    const int32_t *count;
    void *O;
    float *LSE;
    int32_t *dev_err;
    msa_mode mode;                /* PREFILL (0) or CHUNK */
    const int32_t *seq_pt;        /* chunk */
    int64_t max_pages;            /* chunk */
    int64_t num_pages;            /* chunk */
    const int32_t *q_pos;         /* chunk */
} msa_prefill_args;

size_t msa_sparse_attn_prefill_workspace_size(const msa_prefill_args *args, int64_t chunk_queries);
msa_status msa_sparse_attn_prefill(const msa_prefill_args *args, void *ws, size_t ws_bytes,
                                   msa_stream_t stream);

/* --------------------------------------------------------------------------
 * a5-a6. Sparse attention, paged decode
 *
 * One query token per sequence.  Row r = b * Hkv + g of the flattened page
 * table (msa_build_page_table) lists the row's selected pages; the G query
 * heads of group g attend to the first n[r] pages, the last of which holds
 * last_len[r] valid tokens ([serving], "MSA con paged attention").  Each
 * (row, page) pair is an independent split of the softmax; the partials go to
 * the workspace and the CTA that finishes a row's last split combines them with
 * the log-sum-exp merge.
 *     Q [B, Hq, D] bf16 strides (b, h); K_pool, V_pool [num_pages, Hkv, Bk, D]
 *     bf16 with common strides kv_stride = (page, g, t);
 *     pt [B*Hkv, k], n [B*Hkv], last_len [B*Hkv] int32;
 *     O [B, Hq, D] bf16 (dense), LSE [B, Hq] fp32 (dense).
 * Workspace: msa_sparse_attn_decode_workspace_size(args) bytes (fp32 partial
 * outputs and LSEs and one counter per row: B*Hq*k*(D+1)*4 + B*Hkv*4 + 256
 * bytes; the B*Hkv int32 counters start at byte B*Hq*k*(D+1)*4).
 * scratch_zeroed = 0: the call clears the counters first (one memset on the
 * stream).  scratch_zeroed = 1: the caller guarantees they are zero (a
 * zero-filled workspace, or one left by a previous call with the same B, Hq,
 * Hkv, k and D) and the memset is skipped.  Either way a call that raises no
 * device error leaves the counters zero; after one that does, zero them again
 * (or pass 0).  Page ids outside [0, num_pages) are skipped
 * (MSA_DEVERR_BAD_PAGE).  softmax_scale <= 0 selects 1/sqrt(D).  Pool slots
 * past a row's last_len must hold finite values (a zero-filled pool does).
 * ------------------------------------------------------------------------ */
typedef struct msa_decode_args {
    int B, Hq, Hkv, D, Bk, k;
    float softmax_scale;
    const void *Q;
    int64_t Q_stride[2];
    const void *K_pool;
    const void *V_pool;
    int64_t kv_stride[3];
    int64_t num_pages;
    const int32_t *pt;
    const int32_t *n;
    const int32_t *last_len;
    void *O;
    float *LSE;
    int32_t *dev_err;
    int scratch_zeroed;
} msa_decode_args;

size_t msa_sparse_attn_decode_workspace_size(const msa_decode_args *args);
msa_status msa_sparse_attn_decode(const msa_decode_args *args, void *ws, size_t ws_bytes,
                                  msa_stream_t stream);

/* --------------------------------------------------------------------------
 * Paged decode attention without caller-provided scratch.
 *
 * The MSA pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory or pass a workspace: a serving loop whose
 * allocator is frozen after start-up, a plug-in whose host framework owns every
 * device allocation, or code running where an allocation could synchronise the
 * device.  It computes exactly what msa_sparse_attn_decode computes, with the
 * same arguments and checks, but keeps its partial outputs in one array of
 * MSA_NOALLOC_SCRATCH_BYTES that is part of the library's device image and
 * stays resident on every device that loads the library until the process
 * exits.  It allocates nothing and frees nothing.
 *   - Sizes whose scratch, B*Hq*k*(D+1)*4 + B*Hkv*4 + 256 bytes, exceeds the array are
 *     rejected with MSA_ERR_WORKSPACE and a message; use msa_sparse_attn_decode
 *     with a workspace for those.
 *   - The first call on a device looks up the array's device address with that
 *     device current, and so does the first call after the device's context
 *     was destroyed and created again (cudaDeviceReset); make such a call
 *     before any stream capture.  A lookup that fails returns MSA_ERR_CUDA
 *     and is tried again by the next call.
 *   - All calls share the array, which keeps the last call's contents.  Calls
 *     whose kernels overlap on the GPU (other streams, other host threads)
 *     race on it: serialise them.  Each call clears the per-row counters it
 *     needs (scratch_zeroed is ignored) and writes every partial the merge
 *     reads before reading it.
 * ------------------------------------------------------------------------ */
#define MSA_NOALLOC_SCRATCH_BYTES (32u << 20)

msa_status msa_sparse_attn_decode_noalloc(const msa_decode_args *args, msa_stream_t stream);

/* --------------------------------------------------------------------------
 * Dense comparator: paged decode over every cached token
 *
 * The pages quote MSA's speed only against dense attention ("MiniMax M3: Como
 * la atencion dispersa hace practicos a los agentes de largo alcance", bullet
 * "Rapido en produccion": 14.2x prefill and 7.6x decode on H800; the M2-report
 * article, section "MiniMax Sparse Attention (MSA) y escalado subcuadratico
 * entrante": 9.7x / 15.6x at 1M tokens).  This call is that baseline for a
 * decode step, on the same inputs and layouts as the MSA decode step but with
 * no index branch and no selection: each query attends to all L_b tokens of
 * its sequence, what MSA computes when k covers every block.
 *     O[b, h] = sum_{t < L_b} softmax_t(scale * Q[b, h] . K[b, g, t]) V[b, g, t],
 *     g = h / G, logical block j of sequence b in page seq_pt[b][j];
 *     LSE[b, h] = ln sum_t exp(scale * Q[b, h] . K[b, g, t]).
 *     Q [B, Hq, D] bf16 strides (b, h); K_pool, V_pool [num_pages, Hkv, Bk, D]
 *     bf16 with common strides kv_stride = (page, g, t); seq_pt [B, max_pages]
 *     and seq_len [B] int32; O [B, Hq, D] bf16 (dense), LSE [B, Hq] fp32
 *     (dense, may be NULL).
 * Workspace: msa_dense_attn_decode_workspace_size(args) bytes of caller
 * scratch (per-split partials and one page counter per (b, g) row, the
 * counters last).  scratch_zeroed works as in msa_sparse_attn_decode.
 * A sequence whose length is outside [1, max_pages * Bk] gets O = 0 and
 * LSE = -inf and raises MSA_DEVERR_BAD_LEN; a page id outside [0, num_pages)
 * is not read (MSA_DEVERR_BAD_PAGE) and its tokens are left out.  Pool slots
 * past a sequence's last token must hold finite values.  B <= 1024 and
 * B * Hkv * max_pages < 2^30.
 * ------------------------------------------------------------------------ */
typedef struct msa_dense_decode_args {
    int B, Hq, Hkv, D, Bk;
    float softmax_scale;
    const void *Q;
    int64_t Q_stride[2];
    const void *K_pool;
    const void *V_pool;
    int64_t kv_stride[3];
    int64_t num_pages;
    const int32_t *seq_pt;
    int64_t max_pages;
    const int32_t *seq_len;
    void *O;
    float *LSE;
    int32_t *dev_err;
    int scratch_zeroed;
} msa_dense_decode_args;

size_t msa_dense_attn_decode_workspace_size(const msa_dense_decode_args *args);
msa_status msa_dense_attn_decode(const msa_dense_decode_args *args, void *ws, size_t ws_bytes,
                                 msa_stream_t stream);

/* --------------------------------------------------------------------------
 * Dense comparator: causal prefill over every earlier token
 *
 * The prefill half of the same baseline (pages and passages as for
 * msa_dense_attn_decode): exact causal GQA attention with no index branch and
 * no selection, what MSA computes when k covers every block.
 *     O[b, i, h] = sum_{t <= i} softmax_t(scale * Q[b, i, h] . K[b, t, g]) V[b, t, g],
 *     LSE[b, i, h] = ln sum_{t <= i} exp(scale * Q[b, i, h] . K[b, t, g]),  g = h / G.
 *     Q [B, S, Hq, D] bf16 strides (b, s, h); K, V [B, S, Hkv, D] bf16 strides
 *     (b, s, g); O [B, S, Hq, D] bf16 (dense), LSE [B, S, Hq] fp32 (dense, may
 *     be NULL).
 * No workspace.  softmax_scale <= 0 selects 1 / sqrt(D).  B * S < 2^31.
 * ------------------------------------------------------------------------ */
typedef struct msa_dense_prefill_args {
    int B, S, Hq, Hkv, D;
    float softmax_scale;
    const void *Q;
    int64_t Q_stride[3];
    const void *K;
    int64_t K_stride[3];
    const void *V;
    int64_t V_stride[3];
    void *O;
    float *LSE;
    int32_t *dev_err;
} msa_dense_prefill_args;

msa_status msa_dense_attn_prefill(const msa_dense_prefill_args *args, msa_stream_t stream);

/* --------------------------------------------------------------------------
 * a6. Log-sum-exp merge of partial softmax results
 *
 * Partial outputs over blocks recombined by a final log-sum-exp reduction
 * ([serving], "KV-Block-Major"):
 *     LSE[r] = ln sum_p exp(LSE_part[r][p])
 *     O[r]   = sum_p exp(LSE_part[r][p] - LSE[r]) * O_part[r][p]
 * Parts with LSE_part = -inf are empty and skipped (their O_part is not read);
 * a row with no non-empty part gets O = 0 and LSE = -inf.
 *     O_part [rows, parts, D] fp32, LSE_part [rows, parts] fp32 (dense);
 *     O [rows, D] bf16 (dense), LSE [rows] fp32 (may be NULL).
 * D must be a multiple of 4 and at most 512; parts at most 64.
 * ------------------------------------------------------------------------ */
msa_status msa_lse_merge(const float *O_part, const float *LSE_part, int64_t rows, int parts,
                         int D, void *O, float *LSE, int32_t *dev_err, msa_stream_t stream);

/* --------------------------------------------------------------------------
 * Cache append: the step before a decode step
 *
 * Writes each sequence's current token into the 128-token paged caches that
 * index scoring and attention read ([serving], "MSA con paged attention":
 * fixed-size pages; the current token's K, V and index key are in the cache
 * before the step).  For sequence b of length L_b (the new token at position
 * L_b - 1), page = seq_pt[b][(L_b - 1) / Bk], t = (L_b - 1) % Bk, and every
 * KV group g:
 *     K_pool[page, g, t, :]    = K_new[b, g, :]
 *     V_pool[page, g, t, :]    = V_new[b, g, :]
 *     kidx_pool[page, g, t, :] = kidx_new[b, g, :]
 *     K_new, V_new [B, Hkv, D] bf16 strides (b, g); kidx_new [B, Hkv, dI] bf16
 *     strides (b, g); pools as in msa_sparse_attn_decode / msa_index_score
 *     (element strides (page, g, t)); seq_pt [B, max_pages], seq_len [B].
 * A sequence whose length is outside [1, max_pages * Bk] (MSA_DEVERR_BAD_LEN)
 * or whose page id is outside [0, num_pages) (MSA_DEVERR_BAD_PAGE) is not
 * written.  Pointers and strides must be 16-byte aligned; D and dI multiples of 8.
 * A kidx_pool group stride of 0 (one index-key pool shared by the KV groups,
 * as msa_index_score accepts) stores the index key of group 0 only.
 * T > 1 appends T tokens per sequence (a prefill chunk, or draft tokens before
 * a CHUNK-mode call): K_new, V_new [B, T, Hkv, D] and kidx_new [B, T, Hkv, dI]
 * with the (b, g) strides above and token strides new_t_stride = (K_new,
 * V_new, kidx_new); token u of sequence b goes to position L_b - T + u.  A
 * sequence with L_b < T or L_b > max_pages * Bk is not written
 * (MSA_DEVERR_BAD_LEN); a token whose page id is outside [0, num_pages) is
 * not written (MSA_DEVERR_BAD_PAGE).  T = 0 means 1.
 * ------------------------------------------------------------------------ */
typedef struct msa_append_args {
    int B, Hkv, D, dI, Bk;
    const void *K_new;
    int64_t K_new_stride[2];
    const void *V_new;
    int64_t V_new_stride[2];
    const void *kidx_new;
    int64_t kidx_new_stride[2];
    void *K_pool;
    void *V_pool;
    int64_t kv_stride[3];
    void *kidx_pool;
    int64_t kidx_stride[3];
    int64_t num_pages;
    const int32_t *seq_pt;
    int64_t max_pages;
    const int32_t *seq_len;
    int32_t *dev_err;
    int T;                        /* tokens per sequence (0 or 1: one) */
    int64_t new_t_stride[3];      /* T > 1: token strides of K_new, V_new, kidx_new */
} msa_append_args;

msa_status msa_cache_append(const msa_append_args *args, msa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H */
