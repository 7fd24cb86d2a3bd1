/*
 * csa2.h -- C ABI of the CSA2 global-attention decode path on GB300 (sm_103a).
 *
 * The path (DeepSeek-V4.1-Flash, "An infra-oriented diagram of the
 * DeepSeek-V4.1-Flash architecture", reading notes; perchy.ai card
 * "Full. Reindex. Reuse."):
 *   1. lightning-indexer score of every visible cache entry      csa2_index_score
 *   2. top-512 selection (or a 2,048-block candidate pool first)  csa2_topk
 *   3. dequantisation of the selected FP4 latents + 64-head MQA
 *      attention over them and the 128-token FP8 window          csa2_sparse_attn
 *   0. cache write: FP4 / FP8 packing (m=1 or gated m=2)          csa2_fp4_pack
 *
 * Conventions (every entry point):
 *   - Returns a csa2_status.  Nothing aborts, prints or allocates device memory.
 *   - Pointers marked (device) are caller-owned device buffers; the library
 *     never frees or retains them.  Scratch space is passed in by the caller;
 *     csa2_workspace_size() says how much.
 *   - All work is enqueued on `stream` and is asynchronous.  Host-side argument
 *     checks happen before anything is launched; on a failed check nothing is
 *     launched and CSA2_ERR_INVALID_ARG / CSA2_ERR_UNSUPPORTED is returned.
 *   - Values held in device arrays (sequence ids, lengths, selected indices,
 *     pool block ids) are checked by the kernels: an out-of-range value is
 *     skipped and records CSA2_ERR_BOUNDS in a sticky device status word, read
 *     (and cleared) with csa2_get_device_status().  No kernel traps or spins
 *     without a bound.
 *   - Errors from the CUDA runtime (launch failures) return CSA2_ERR_CUDA.
 *
 * Cache record formats (logical bytes per record are fixed by the pages; the
 * physical arrangement below is this library's choice):
 *   KV  (S1) 288 B per entry, array of records [n_seq][n_max][288]: bytes 0..255
 *            hold 512 FP4 E2M1 codes (low nibble = even channel), bytes
 *            256..287 hold 32 E4M3 scales, one per 16 channels (the study's
 *            section "The KV cache" sizes a main-cache entry at 288 bytes: 512
 *            FP4 codes and one E4M3 scale for each 16 channels).
 *   IDX (S2) 68 B per entry as two planes, so that every row is 16-B aligned:
 *            nibbles [rows][64] (128 E2M1 codes) and scales [rows][4] (E8M0, one
 *            per 32 channels) (the same section sizes an indexer key at 68
 *            bytes: 128 FP4 codes, an E8M0 scale for each 32).  The nibble plane is stored in the
 *            64-byte swizzled order of the tensor cores: the 16-byte chunk c
 *            (channels 32c .. 32c+31) of a row at byte address A is stored at
 *            chunk c ^ ((A >> 7) & 3) of that row; with a 512-B aligned plane
 *            that is c ^ ((row >> 1) & 3).  csa2_fp4_pack writes this order, so
 *            any 8-row-aligned range can be packed independently.  The indexer
 *            query heads (S4) use the same format with rows = n_q * 32.
 *   SWA (S3) 528 B per entry [n_seq][swa_cap][528]: 512 E4M3 values then 16
 *            E8M0 scales, one per 32 channels (a reading of the same section,
 *            which gives the window as 128 FP8 entries of 528 bytes).
 *
 * Rounding (shared by every packer): round to nearest, ties to even, saturating
 * at the format's largest finite value; the sign of x is kept when the magnitude
 * rounds to zero.  E4M3 latent scale = E4M3(amax/6); a group whose scale is zero
 * stores zero codes.  E8M0 scale = the smallest power of two >= amax/6 (FP4) or
 * >= amax/448 (FP8), exponent clamped to [-127, 127]; amax = 0 stores byte 0 and
 * zero codes.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *csa2_stream_t;   /* == cudaStream_t; NULL = legacy default stream */

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,   /* a null pointer, a negative or misaligned size, an unknown kind */
  CSA2_ERR_UNSUPPORTED = 2,   /* parameters other than the pages' constants, k above the limit */
  CSA2_ERR_CUDA = 3,          /* the CUDA runtime reported an error                           */
  CSA2_ERR_BOUNDS = 4,        /* (device) an index or length in a device array was out of range */
  CSA2_ERR_TIMEOUT = 5,       /* (device) a bounded wait ran out                               */
  CSA2_ERR_WORKSPACE = 6      /* the workspace passed in is smaller than required             */
} csa2_status;

/* Record kinds for csa2_entry_bytes / csa2_fp4_pack. */
enum { CSA2_KV_NVFP4 = 0, CSA2_IDX_MXFP4 = 1, CSA2_SWA_MXFP8 = 2 };
/* Output dtypes for csa2_sparse_attn. */
enum { CSA2_OUT_BF16 = 0, CSA2_OUT_F32 = 1 };
/* Operations for csa2_workspace_size. */
enum { CSA2_OP_TOPK = 0, CSA2_OP_SPARSE_ATTN = 1, CSA2_OP_DECODE = 2, CSA2_OP_DECODE_HOST = 3, CSA2_OP_DECODE_MQ = 4,
       CSA2_OP_BUILD_CACHE = 5, CSA2_OP_DECODE_REINDEX = 6 };

/* Model constants.  The kernels are built for the pages' values only
 * (study, reading notes: 64 heads, 512-wide latent, RoPE on 64 of the 512
 * dims; lightning indexer 32 x 128, top-512; pool of 2,048 blocks of 8;
 * helix.ml: 128-token window).  rope_base and sm_scale are free. */
typedef struct {
  int heads;        /* 64                      */
  int dim;          /* 512                     */
  int rope_dim;     /* 64                      */
  int rope_off;     /* 448 (dims 448..511)     */
  double rope_base; /* 10000                   */
  float sm_scale;   /* 1/sqrt(512)             */
  int idx_heads;    /* 32                      */
  int idx_dim;      /* 128                     */
  int topk;         /* 512                     */
  int swa;          /* 128                     */
  int block;        /* 8                       */
  int pool_blocks;  /* 2048                    */
} csa2_params;

/* Fills *p with the pages' constants.  Never fails for a non-null p. */
csa2_status csa2_default_params(csa2_params *p);

/* Bytes per logical record: KV 288, IDX 68, SWA 528; 0 for an unknown kind. */
size_t csa2_entry_bytes(int kind);

/* Human-readable name of a status code (static string). */
const char *csa2_status_string(csa2_status s);

/*
 * csa2_fp4_pack -- cache write: quantise bf16 rows into cache records.
 * (An infra-oriented diagram of the DeepSeek-V4.1-Flash architecture, reading
 * notes and section "The KV cache": the encoder pools each pair of tokens into
 * one entry through a learned softmax gate, and the latent cache holds E2M1
 * values with an E4M3 scale for every 16 channels.)
 *
 *   kind         CSA2_KV_NVFP4 (src rows of 512), CSA2_IDX_MXFP4 (rows of 128),
 *                CSA2_SWA_MXFP8 (rows of 512).
 *   src          (device) bf16 [rows][width], row-major, 16-B aligned.
 *   rows         number of source rows (tokens); >= 0.  0 launches nothing.
 *   m            1, or 2 (KV only): rows must be even; output row r pools
 *                source rows 2r and 2r+1 per channel with weights
 *                softmax(gate_logits[2r][c], gate_logits[2r+1][c]), computed
 *                in fp64 and rounded to bf16 before packing.
 *   gate_logits  (device) fp32 [rows][512] when m == 2, else must be NULL.
 *   dst          (device) KV/SWA: rows/m records of 288/528 B; IDX: the nibble
 *                plane [rows][64].  16-B aligned.
 *   dst_scales   (device) IDX only: the scale plane [rows][4]; NULL otherwise.
 */
csa2_status csa2_fp4_pack(int kind, const void *src, int64_t rows, int m, const float *gate_logits,
                          void *dst, void *dst_scales, csa2_stream_t stream);

/*
 * csa2_index_score -- lightning-indexer scores.
 * (An infra-oriented diagram of the DeepSeek-V4.1-Flash architecture, reading
 * notes: the indexer compares 32 FP4 query heads of width 128 with the single
 * key of each entry, clamps each head's dot product at zero and adds them up
 * with one weight per head):
 *     s_j = sum_{h<32} w_h * max(0, qhat_h . khat_j)
 * with qhat, khat the dequantised FP4 values (E2M1 x E8M0), fp32 accumulation.
 *
 *   key_nib, key_scale  (device) IDX cache planes of n_seq * n_max entries;
 *                       entry j of sequence b is row b*n_max + j.  key_nib
 *                       512-B aligned, key_scale 16-B aligned.
 *   n_max               entries per sequence; a positive multiple of 128.
 *   n_seq               number of sequences (>= 1).
 *   q_nib, q_scale      (device) indexer queries, IDX format, rows = n_q*32;
 *                       q_nib 512-B aligned, q_scale 16-B aligned.
 *   w                   (device) fp32 [n_q][32] per-head weights, 16-B aligned.
 *   q_seq               (device) int32 [n_q] sequence of each query.
 *   n_vis               (device) int32 [n_q]: entries [0, n_vis) are visible.
 *   n_q                 number of queries (0 launches nothing).
 *   pool_blocks         NULL: Full mode, scores[q][j] for j < n_vis[q] (other
 *                       columns untouched).  Non-NULL (device) int32 [n_q][2048]
 *                       block ids (-1 = none): Reindex mode, scores[q][s] for the
 *                       16,384 pool slots s (entry 8*pool_blocks[q][s/8] + s%8),
 *                       -inf for a slot whose block is -1 or whose entry is not
 *                       visible (same page, lightning-indexer note: decoder
 *                       Reindex layers score only the 16,384 positions of the
 *                       pool an earlier layer picked as 2,048 blocks of 8).
 *   scores              (device) fp32, row stride score_stride (>= n_max in Full
 *                       mode, >= 16384 in Reindex mode).
 */
csa2_status csa2_index_score(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq,
                             const void *q_nib, const void *q_scale, const float *w,
                             const int32_t *q_seq, const int32_t *n_vis, int n_q,
                             const int32_t *pool_blocks, float *scores, int64_t score_stride,
                             const csa2_params *params, csa2_stream_t stream);

/*
 * csa2_topk -- top-k selection by (score descending, index ascending): the lower
 * index wins ties; -0.0 equals +0.0.  Output indices ascending, padded with -1
 * when fewer than k items are valid.
 * (perchy.ai/models/deepseek, card "Full. Reindex. Reuse.": the main selection
 * keeps 512 entries and later decoder indexers look at no more than 16,384
 * candidates; An infra-oriented diagram of the DeepSeek-V4.1-Flash architecture,
 * lightning-indexer note: those candidates are 2,048 blocks of 8 entries.)
 *
 *   scores        (device) fp32 [n_q][score_stride].
 *   n_valid       (device) int32 [n_q]: number of visible entries.
 *   n_max         entries per row considered (Full mode: columns [0, n_max);
 *                 <= score_stride).
 *   k             1 .. 2048.
 *   block         1: items are entries j < n_valid.
 *                 8: items are blocks b of 8 entries (b*8 < n_valid), scored by
 *                    the max over their visible entries (a reading of the
 *                    card's selection in 8-entry blocks); the output holds block
 *                    ids.  pool_blocks must be NULL.
 *   pool_blocks   NULL, or (device) int32 [n_q][2048] when the scores are Reindex
 *                 pool slots (row length 16384): item s is entry
 *                 8*pool_blocks[q][s/8] + s%8, valid if the block id is >= 0 and
 *                 the entry < n_valid; the output holds those entry indices.
 *   out           (device) int32 [n_q][k].
 *   workspace     (device) scratch of at least csa2_workspace_size(CSA2_OP_TOPK,..)
 *                 bytes, 256-B aligned; contents need no initialisation.
 */
csa2_status csa2_topk(const float *scores, int64_t score_stride, int n_q, const int32_t *n_valid,
                      int64_t n_max, int k, int block, const int32_t *pool_blocks, int32_t *out,
                      void *workspace, size_t workspace_bytes, csa2_stream_t stream);

/*
 * csa2_sparse_attn -- 64-head MQA attention over the selected entries plus the
 * sliding window, k = v.
 * (An infra-oriented diagram of the DeepSeek-V4.1-Flash architecture, reading
 * notes: each token has one 512-wide latent serving as both key and value for
 * all 64 query heads; attention covers the selected 512 entries plus the
 * window; RoPE acts on 64 of the 512 dimensions and is undone on the output.
 * DeepSeek V4.1 Flash: Why Its Encoder, Engram and KV Cache Matter, section
 * "CSA2 makes long context cheaper to retain": the window is the last 128
 * tokens.)  For each query and head h:
 *     l_i = sm_scale * q_h . khat_i  over i in {selected} + {window}
 *     o_h = sum_i softmax(l)_i khat_i
 * then the pairs (rope_off + 2i, rope_off + 2i + 1), i < 32, are rotated by
 * -pos:  (a, b) <- (a cos t + b sin t, -a sin t + b cos t),
 * t = pos * rope_base^(-2i/64).  A query with no entry at all gets zeros.
 * Arithmetic: dequantised latents are exact (f16 for chunks of selected
 * entries only, bf16 for chunks holding window entries), products accumulate
 * in fp32, and the softmax numerators are rounded to f16 (11 bits) or kept as
 * bf16 hi + lo parts; the row-normalised error against an fp64 evaluation is
 * about 2e-4 (under 2e-3).
 *
 *   q            (device) bf16 [n_q][64][512] (already rotated by upstream).
 *   kv_cache     (device) KV records [n_seq][n_max][288].
 *   sel          (device) int32 [n_q][sel_stride]: entry indices (< n_max) or -1;
 *                sel_stride in 1 .. 512.
 *   swa_cache    (device) SWA records [n_seq][swa_cap][528]; may be NULL when
 *                swa_cap == 0.
 *   q_seq, pos   (device) int32 [n_q]: sequence id, RoPE position of the query.
 *   swa_first, swa_cnt  (device) int32 [n_q]: the window is ring slots
 *                (swa_first + t) % swa_cap, t < swa_cnt, with
 *                0 <= swa_cnt <= min(128, swa_cap) and 0 <= swa_first < swa_cap
 *                when swa_cnt > 0; a query breaking this (or with q_seq out of
 *                range) records CSA2_ERR_BOUNDS and gets zeros.
 *   out          (device) [n_q][64][512], bf16 or fp32 per out_dtype.
 *   workspace    (device) >= csa2_workspace_size(CSA2_OP_SPARSE_ATTN, ..) bytes.
 */
csa2_status csa2_sparse_attn(const void *q, const void *kv_cache, int64_t n_max, int n_seq,
                             const int32_t *sel, int sel_stride, const void *swa_cache, int swa_cap,
                             const int32_t *q_seq, const int32_t *pos, const int32_t *swa_first,
                             const int32_t *swa_cnt, int n_q, void *out, int out_dtype,
                             const csa2_params *params, void *workspace, size_t workspace_bytes,
                             csa2_stream_t stream);

/*
 * csa2_decode -- one Full-layer decode step: csa2_index_score over every
 * visible entry, top-512 selection, csa2_sparse_attn over the selection and
 * the window, issued as one call.  The pages give no such call; it composes
 * the three steps above (same arguments, same meaning, the same selection as
 * the chain csa2_index_score -> csa2_topk(k = 512, block = 1) ->
 * csa2_sparse_attn(sel_stride = 512)), and lets the indexer's epilogue also
 * write the maxima the selection starts from, which saves the selection's
 * first pass over the scores.  For small batches (up to about 30 queries on
 * 152 SMs) over long rows, the selection also hands its candidates (a superset
 * of the selected entries, at most 640, in index order) to the attention before
 * its exact pass, and the attention masks those below the smallest selected
 * key: the output then attends to exactly the selected entries and the window,
 * but groups them into other chunks than csa2_sparse_attn does, so it agrees
 * with the chain's to rounding (relative 1e-3) rather than bit for bit; the
 * same holds for batches (about 39 to 76 queries on 152 SMs) where the
 * attention runs a query's window chunk first in its last split, while the
 * selection finishes.  The same inputs give the same bits on every call.
 *
 *   key_nib .. n_q      as csa2_index_score (Full mode; scores are kept in the
 *                       workspace).
 *   q .. swa_cnt, out, out_dtype, params   as csa2_sparse_attn.
 *   sel                 (device) int32 [n_q][512]: the selected entries
 *                       (ascending, -1 padding), as csa2_topk writes them.
 *   workspace           (device) >= csa2_workspace_size(CSA2_OP_DECODE, n_q,
 *                       n_max, 512) bytes, 256-B aligned; no initialisation.
 */
csa2_status csa2_decode(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq, const void *q_nib,
                        const void *q_scale, const float *w, const int32_t *q_seq, const int32_t *n_vis, int n_q,
                        const void *q, const void *kv_cache, const void *swa_cache, int swa_cap, const int32_t *pos,
                        const int32_t *swa_first, const int32_t *swa_cnt, int32_t *sel, void *out, int out_dtype,
                        const csa2_params *params, void *workspace, size_t workspace_bytes, csa2_stream_t stream);

/*
 * csa2_decode_reindex -- the decode step of a Reindex layer ("An
 * infra-oriented diagram of the DeepSeek-V4.1-Flash architecture", reading
 * notes on the Full / Reindex / Reuse roles; perchy.ai card "Full. Reindex.
 * Reuse."): the layer's own indexer query scores the 16,384 positions of the
 * candidate pool the Full layer chose (2,048 blocks of 8), the top-512 of the
 * pool is selected, and the attention runs over it and the window, as one
 * call.  The results are those of the chain csa2_index_score (pool mode) ->
 * csa2_topk(k = 512, block = 1, pool_blocks) -> csa2_sparse_attn(sel_stride =
 * 512): the selection bit for bit, the output bit for bit where the attention
 * splits a query's chunks as csa2_sparse_attn does, else to rounding (relative
 * 1e-3; for some batch sizes the call runs a query's window chunk first in its
 * last split, while the selection finishes).  Inside the call the indexer also
 * writes the largest order key of every 8-entry block of the pool, so that
 * the selection reads only the blocks that can hold one of the 512, and the
 * attention, whose inputs are final before the call starts, stages them while
 * the selection runs.
 *
 *   key_nib .. n_q      as csa2_index_score; q_nib, q_scale, w are the
 *                       Reindex layer's indexer query and weights.
 *   pool_blocks         (device) int32 [n_q][2048]: the pool's block ids, as
 *                       csa2_topk(block = 8) writes them (-1: none).
 *   q .. swa_cnt, out, out_dtype, params   as csa2_sparse_attn.
 *   sel                 (device) int32 [n_q][512]: the selected entries
 *                       (ascending, -1 padding), as csa2_topk writes them.
 *   workspace           (device) >= csa2_workspace_size(CSA2_OP_DECODE_REINDEX,
 *                       n_q, n_max, 512) bytes, 256-B aligned; no initialisation.
 */
csa2_status csa2_decode_reindex(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq,
                                const void *q_nib, const void *q_scale, const float *w, const int32_t *q_seq,
                                const int32_t *n_vis, int n_q, const int32_t *pool_blocks, const void *q,
                                const void *kv_cache, const void *swa_cache, int swa_cap, const int32_t *pos,
                                const int32_t *swa_first, const int32_t *swa_cnt, int32_t *sel, void *out,
                                int out_dtype, const csa2_params *params, void *workspace, size_t workspace_bytes,
                                csa2_stream_t stream);

/*
 * csa2_index_score_mq -- csa2_index_score (Full mode) for groups of queries
 * that share a sequence, such as several draft positions of one sequence
 * decoded in the same step (DeepSeek V4.1 Flash: Why Its Encoder, Engram and
 * KV Cache Matter, section on DSpark: five future positions per step).  The
 * queries [g * q_group, g * q_group + q_group) must all name the same
 * sequence; each of its key units is read once for the whole group and
 * multiplied with all 32 x q_group query heads at once.  Results as
 * csa2_index_score for every query (scores[q][j] for j < n_vis[q]).
 *
 *   q_group    1 .. 6; n_q a multiple of q_group.  A group whose queries name
 *              different sequences (or an out-of-range sequence or length) is
 *              skipped and records CSA2_ERR_BOUNDS.
 *   the rest   as csa2_index_score (no pool mode).
 */
csa2_status csa2_index_score_mq(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq,
                                const void *q_nib, const void *q_scale, const float *w, const int32_t *q_seq,
                                const int32_t *n_vis, int n_q, int q_group, float *scores, int64_t score_stride,
                                const csa2_params *params, csa2_stream_t stream);

/*
 * csa2_decode_mq -- the decode step of csa2_decode for groups of q_group
 * queries per sequence: csa2_index_score_mq, then the top-512 of every query
 * (csa2_topk), then csa2_sparse_attn of every query; the results are those of
 * that chain.  Arguments as csa2_decode, with q_group as in
 * csa2_index_score_mq; workspace >= csa2_workspace_size(CSA2_OP_DECODE_MQ,
 * n_q, n_max, 512) bytes, 256-B aligned, no initialisation.
 */
csa2_status csa2_decode_mq(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq, const void *q_nib,
                           const void *q_scale, const float *w, const int32_t *q_seq, const int32_t *n_vis, int n_q,
                           int q_group, const void *q, const void *kv_cache, const void *swa_cache, int swa_cap,
                           const int32_t *pos, const int32_t *swa_first, const int32_t *swa_cnt, int32_t *sel,
                           void *out, int out_dtype, const csa2_params *params, void *workspace,
                           size_t workspace_bytes, csa2_stream_t stream);

/*
 * csa2_decode_host -- csa2_decode with the step's inputs and outputs in host
 * memory: the end-to-end call of a decode step.  The caches (indexer keys,
 * latents, window) stay resident in device memory; the per-step tensors
 * travel with the call.  On `stream`, in order: the inputs into the
 * workspace -- where all four input buffers are page-locked (cudaHostAlloc,
 * cudaMallocHost, cudaHostRegister: device-accessible under unified
 * addressing), one kernel reads them in place and packs the indexer query;
 * otherwise one cudaMemcpyAsync per buffer and csa2_fp4_pack --, then
 * csa2_decode, whose last grid writes the output straight into h_out where
 * that is page-locked (else into the workspace, then one cudaMemcpyAsync),
 * then one cudaMemcpyAsync into h_sel, if given.  Either way the results are
 * the same.  Asynchronous: the host buffers must stay valid
 * and unchanged (and the outputs unread) until the stream has passed the
 * call; pageable memory works but serialises the copies.
 *
 *   key_nib .. n_seq, kv_cache, swa_cache, swa_cap   (device) as csa2_decode.
 *   h_q        (host) bf16 [n_q][64][512], the attention query (rotated).
 *   h_qidx     (host) bf16 [n_q][32][128], the indexer query before packing.
 *   h_w        (host) fp32 [n_q][32], the indexer head weights.
 *   h_desc     (host) int32 [5][n_q]: rows q_seq, n_vis, pos, swa_first,
 *              swa_cnt (meanings as csa2_decode).
 *   h_sel      (host, may be NULL) int32 [n_q][512]: receives the selection.
 *   h_out      (host) [n_q][64][512], bf16 or fp32 per out_dtype.
 *   workspace  (device) >= csa2_workspace_size(CSA2_OP_DECODE_HOST, n_q,
 *              n_max, 512) bytes, 256-B aligned; no initialisation.
 * Argument checks and errors as csa2_decode; a failed copy returns
 * CSA2_ERR_CUDA.
 */
csa2_status csa2_decode_host(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq, const void *kv_cache,
                             const void *swa_cache, int swa_cap, const void *h_q, const void *h_qidx, const float *h_w,
                             const int32_t *h_desc, int n_q, int32_t *h_sel, void *h_out, int out_dtype,
                             const csa2_params *params, void *workspace, size_t workspace_bytes, csa2_stream_t stream);

/*
 * csa2_index_key_proj -- the indexer keys of cache entries: the 512 -> 128
 * projection of each entry's latent ("An infra-oriented diagram of the
 * DeepSeek-V4.1-Flash architecture", reading notes on the Full layer's global
 * KV: the indexer's key is a 512 -> 128 projection of the same latent).  The
 * pages give no weights; the caller supplies them.
 *   keys[r][n] = bf16( sum_c latent[r][c] * w_idx[n][c] ), fp32 accumulation on
 *   the tensor cores, rounded to nearest even.
 *   latent  (device) bf16 [rows][512], 16-B aligned.
 *   w_idx   (device) bf16 [128][512], 16-B aligned.
 *   keys    (device) bf16 [rows][128], 16-B aligned; the input of
 *           csa2_fp4_pack(CSA2_IDX_MXFP4, ...).
 */
csa2_status csa2_index_key_proj(const void *latent, int64_t rows, const void *w_idx, void *keys,
                                csa2_stream_t stream);

/*
 * csa2_build_cache -- the cache entries of a prompt (the study's reading
 * notes: encoder caches pool two tokens into one entry with a learned softmax
 * gate, m = 2; the decoder's Full layer keeps one entry per token, m = 1; the
 * indexer's key is a 512 -> 128 projection of the entry's latent): per entry,
 * the latent (gated pooling for m = 2), its 288-B main-cache record, its key
 * (csa2_index_key_proj) and the key's two-plane 68-B record -- the same bytes
 * as csa2_fp4_pack(CSA2_KV_NVFP4, m), csa2_index_key_proj and
 * csa2_fp4_pack(CSA2_IDX_MXFP4) on the pooled latents.  Prompts of any length
 * (1,048,576 tokens and more) are built in chunks of 131,072 entries, so the
 * scratch stays bounded (168 MB for m = 2, 34 MB for m = 1).
 *   tokens       (device) bf16 [n_tokens][512], 16-B aligned.
 *   n_tokens     a multiple of 8 m (so that chunks start on 8-row boundaries
 *                of the key plane).
 *   m, gate_logits   as csa2_fp4_pack (gate_logits [n_tokens][512] for m = 2,
 *                NULL for m = 1).
 *   w_idx        (device) bf16 [128][512].
 *   kv           (device) [n_tokens / m][288]; idx_nib [n_tokens / m][64]
 *                (512-B aligned, the swizzled key plane); idx_scale
 *                [n_tokens / m][4].  Entry e of the prompt is row e of each.
 *   workspace    (device) >= csa2_workspace_size(CSA2_OP_BUILD_CACHE, 0,
 *                n_tokens, m) bytes, 256-B aligned; no initialisation.
 */
csa2_status csa2_build_cache(const void *tokens, int64_t n_tokens, int m, const float *gate_logits,
                             const void *w_idx, void *kv, void *idx_nib, void *idx_scale, void *workspace,
                             size_t workspace_bytes, csa2_stream_t stream);

/*
 * csa2_profile_events -- measurement hook: while set, csa2_decode and
 * csa2_decode_reindex record `begin` on their stream just before they launch
 * the indexer and `end` just after it, so that the indexer kernel of the step
 * itself (the instantiation that also writes the selection's maxima) can be
 * timed with cudaEventElapsedTime.  Recording between the step's kernels keeps
 * the next kernel from starting early beside the indexer, so a step timed this
 * way runs a little slower than one that is not.  Both null: off.  The setting
 * is per host thread.
 *
 *   begin, end   cudaEvent_t (created by the caller), or both null.
 */
csa2_status csa2_profile_events(void *begin, void *end);

/*
 * csa2_workspace_size -- scratch bytes needed by an operation.
 *   op = CSA2_OP_TOPK:        n_q queries, n_items = items per row (entries,
 *                             blocks, or 16384 pool slots), k.
 *   op = CSA2_OP_SPARSE_ATTN: n_q queries, n_items = sel_stride + 128, k unused.
 *   op = CSA2_OP_DECODE:      n_q queries, n_items = n_max, k unused (512).
 *   op = CSA2_OP_DECODE_HOST: as CSA2_OP_DECODE (the device copies of the
 *                             step's inputs and outputs are included).
 *   op = CSA2_OP_DECODE_MQ:   n_q queries, n_items = n_max, k unused (512).
 *   op = CSA2_OP_BUILD_CACHE: n_q unused, n_items = tokens, k = m (1 or 2).
 *   op = CSA2_OP_DECODE_REINDEX: n_q queries, n_items = n_max, k unused (512).
 * Sizes are for the current device (the attention's split plan follows its
 * SM count).
 */
csa2_status csa2_workspace_size(int op, int n_q, int64_t n_items, int k, size_t *bytes);

/*
 * csa2_topk_noalloc -- csa2_topk for callers that cannot allocate device
 * memory: code running where cudaMalloc is not available or not allowed (inside
 * a host callback or another library's allocation-free region, a plugin whose
 * host owns all device memory, a process that must not grow its footprint after
 * start-up).  The pages have no counterpart of this call: it exists only for
 * the library's users.
 *
 * Same arguments, results and errors as csa2_topk, without the workspace.  The
 * scratch it needs (rows longer than 16,384 items only: 4 bytes per group of
 * scores, 2,048 to 16,384 groups per row; for 1,048,576-entry rows and k = 512
 * that is 8 KiB per query) lives in one fixed device array of
 * CSA2_TOPK_NOALLOC_SCRATCH_BYTES (4 MiB), held on each GPU until the process
 * exits.  With CUDA's default lazy module loading the array is mapped on a
 * device only when its module is first loaded there, i.e. by the first call
 * of this function on that device: that first call grows the device
 * footprint by the 4 MiB.  Callers that need a fixed footprint after start-up
 * make one call on each device (any size) during start-up.  A call whose
 * scratch would exceed it returns CSA2_ERR_WORKSPACE and launches nothing (use
 * csa2_topk with a workspace instead).  The call allocates nothing and calls no
 * allocating routine.  The first call on a device looks up the array's device
 * address on that device; make that first call before any stream capture.
 * All calls share the one array: calls that can run at the same time on the
 * GPU (other streams, other host threads) race and must be serialised by the
 * caller.  Nothing has to be cleared between calls: every scratch value a call
 * reads is written (or cleared) earlier in that same call.
 */
#define CSA2_TOPK_NOALLOC_SCRATCH_BYTES (4u << 20)
csa2_status csa2_topk_noalloc(const float *scores, int64_t score_stride, int n_q, const int32_t *n_valid,
                              int64_t n_max, int k, int block, const int32_t *pool_blocks, int32_t *out,
                              csa2_stream_t stream);

/*
 * csa2_check_bounded_wait -- self-test of the library's bounded waits (the
 * pages have no counterpart).  Launches one warp that takes tensor memory,
 * waits on a barrier that nothing will complete, gives up after limit_us
 * microseconds (1 .. 2,000,000), records CSA2_ERR_TIMEOUT in the device
 * status word, returns the tensor memory and exits: the path every kernel of
 * this library takes when one of its waits runs out (each of them bounded by
 * 2 s of wall time), with nothing asynchronous in flight.  Read the outcome
 * with csa2_get_device_status; the context stays usable.
 */
csa2_status csa2_check_bounded_wait(unsigned limit_us, csa2_stream_t stream);

/*
 * csa2_get_device_status -- synchronises `stream`, returns in *out the first
 * device-side error recorded by any kernel of this library on the current
 * device since the last call (CSA2_OK if none), and clears it.
 */
csa2_status csa2_get_device_status(csa2_stream_t stream, csa2_status *out);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
