/*
 * m3s.h -- C ABI of libm3s: the decode / verify step of indexed (top-k block)
 * sparse attention over a paged NVFP4 (or MXFP4) KV cache, with the cache
 * write optionally fused into the rows' normalisation and rotation,
 * hand-written CUDA for sm_103a.
 *
 * Source of the method: the pull requests "NVFP4 sparse KV" (ROCm/ATOM #2746)
 * and "[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache" (ROCm/ATOM
 * #2744), with the page layout of "MXFP4 KV cache for MiniMax-M3.1 on gfx950"
 * (vllm-project/vllm #64198). Each entry point below names the passage that
 * defines its operation.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Ownership: every pointer argument is caller-owned memory. Tensor
 *    arguments are DEVICE pointers; the library never allocates, frees,
 *    synchronises or reads device data on the host, so every call can be
 *    captured in a CUDA graph. Host-only arguments are passed by value.
 *  - BF16 tensors are passed as their raw 16-bit patterns (uint16_t).
 *  - head_dim is 128 and a page (= a block) holds 128 tokens; these are the
 *    only built values (the pages' guard requires page == 128).
 *  - Every call returns an m3s status. Argument errors are detected on the
 *    host before any launch and nothing is launched.
 *  - Data-dependent errors found on the device (a slot, page or block id out
 *    of range) never fault and are never wrapped: the kernel skips the access
 *    and ORs an M3S_DEVERR_* bit into the caller's int32 error word `err`
 *    (device memory, may be NULL to ignore; it is never cleared by the
 *    library).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). All work
 *    of a call is enqueued on it, in order.
 *  - Alignment: plane, tensor and workspace pointers must be 16-byte aligned;
 *    the BF16 row stride of the store must be a multiple of 8 elements.
 *  - Queries (q, q_idx) may hold any finite BF16 value. The tensor-core
 *    products take f16 operands, so each (row, head) of the queries is scaled
 *    by a power of two 2^-e before its conversion (e = the exponent of the
 *    head's largest magnitude minus 15, so it lands in [2^15, 2^16)) and the
 *    scale is undone exactly in fp32: scores as 2^e_ref times a sum whose
 *    weights carry 2^(e_h - e_ref) (e_ref the row's largest e_h), attention
 *    logits through a per-head logit scale. Elements below 2^-29 of their
 *    head's largest round as f16 subnormals (below 2^-40 they vanish); a weight
 *    whose w_h 2^(e_h - e_ref) falls below fp32's normal range rounds. Results
 *    beyond fp32's range (a block score or logit above ~3.4e38) overflow.
 */
#ifndef M3S_H_
#define M3S_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values) ---- */
#define M3S_OK 0
#define M3S_ERR_INVALID 1     /* null pointer, negative size, misalignment, bad stride */
#define M3S_ERR_UNSUPPORTED 2 /* a shape outside the built bounds (head counts, top-k, ...) */
#define M3S_ERR_WORKSPACE 3   /* ws_bytes below m3s_workspace_bytes() */
#define M3S_ERR_LAUNCH 4      /* the CUDA launch itself failed */

/* ---- device error bits (OR-ed into *err) ---- */
#define M3S_DEVERR_SLOT 1     /* store: slot >= num_pages * 128 (row skipped) */
#define M3S_DEVERR_BLOCK_ID 2 /* attention: a top-k id >= the row's block count or the table width */
#define M3S_DEVERR_PAGE 4     /* a block-table entry outside [0, num_pages) (block skipped) */
#define M3S_DEVERR_ROW 8      /* a row's request outside [0, B) or its length beyond the table */
#define M3S_DEVERR_QRANGE 16  /* a query element that is inf or NaN */
#define M3S_DEVERR_TIMEOUT 32 /* a bounded wait for an asynchronous copy gave up (kernel returned) */

/* ---- limits of this build ---- */
#define M3S_HEAD_DIM 128
#define M3S_PAGE 128
#define M3S_MAX_TOPK 64
#define M3S_MAX_INDEX_HEADS 16
#define M3S_MAX_GQA 16 /* q heads per KV head */

/*
 * A paged FP4 plane pair (the pool of one K, V or index-K tensor).
 * "NVFP4 sparse KV" (ROCm/ATOM #2746), Summary: the pool's k/v and scale fields
 * are uint8 planes; per token and head a 64 B e2m1 payload plus 8 B of E4M3
 * scales. Within a page the payloads of the 128 tokens come first and the
 * scales sit in their own plane (vllm #64198, Claims: [128 x payload][128 x scales]).
 * The MXFP4 record ("[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache"
 * (ROCm/ATOM #2744), Follow-up: MXFP4 caches; vllm #64198, Overview) has the
 * same payload and one E8M0 scale per 32 elements: 68 B per token and head.
 *
 *   codes  : uint8 [num_pages][num_heads][128][64]; byte i of a token holds
 *            element 2i in its low nibble and element 2i+1 in its high nibble;
 *            nibble = sign(bit 3) | e2m1 magnitude code (bits 0-2).
 *   scales : M3S_FMT_NVFP4: uint8 [num_pages][num_heads][128][8]; byte j is the
 *            E4M3 scale of elements 16j .. 16j+15.
 *            M3S_FMT_MXFP4: uint8 [num_pages][num_heads][128][4]; byte j is the
 *            E8M0 scale 2^(byte - 127) of elements 32j .. 32j+31.
 *   format : M3S_FMT_*; a zero-initialised plane is NVFP4. Any other value is
 *            M3S_ERR_INVALID.
 *   A token's slot is page * 128 + position within the page.
 */
#define M3S_FMT_NVFP4 0
#define M3S_FMT_MXFP4 1
typedef struct {
  uint8_t* codes;
  uint8_t* scales;
  int32_t num_pages;
  int32_t num_heads;
  int32_t format;
} m3s_fp4_plane;
typedef m3s_fp4_plane m3s_nvfp4_plane; /* the NVFP4-only name of the same type */

/* ops for m3s_workspace_bytes */
#define M3S_OP_INDEX_SCORE_TOPK 1
#define M3S_OP_VERIFY_SCORE_TOPK 2
#define M3S_OP_SPARSE_ATTENTION 3
#define M3S_OP_INDEX_CANDIDATES 4
#define M3S_OP_INDEX_ATTENTION 5
#define M3S_OP_VERIFY_INDEX_ATTENTION 6

/*
 * Workspace bytes an op needs (device memory the caller provides as `ws`).
 * A pure host function of its arguments; 0 for unknown ops, and 0 for shapes
 * the calls reject with M3S_ERR_UNSUPPORTED before they look at the
 * workspace: more than 8192 tiles (index ops: R > 8192; verify ops:
 * B * ceil(max_q / 8) > 8192).
 *   R rows, B requests, max_blocks = block-table width (bt_stride), Hq / Hkv
 *   q and KV heads, Hi index heads, topk, max_q = the largest rows-per-request
 *   the verify call will see (the cu_q differences).
 * Index / verify (0 when topk is 0), by the tiles of query rows the call
 * scores (index: one tile per row, ntiles = R; verify: tiles of up to 8 rows
 * of one request, ntiles = B * ceil(max_q / 8)):
 *  - ntiles <= 256: the block scores, R * max_blocks fp32 (the call launches the
 *    scorer, then the top-k);
 *  - ntiles > 256: the streaming top-k's state (one launch): one 4-byte ticket
 *    per tile (rounded up to 256 bytes), then candidate lists of topk 8-byte
 *    keys for (ntiles + 255) slots of 1 (index) or 8 (verify) rows, then
 *    (verify) a score scratch of 256 x 8 x max_blocks fp32. This workspace must
 *    read zero when it is first used (zero it once after allocating it); every
 *    call leaves it that way again, so it can be reused call after call, graph
 *    replays included. A call that raised M3S_DEVERR_TIMEOUT may leave tickets
 *    set: zero the workspace again after one.
 * Index attention (decode rows): candidate lists of topk keys for R + 255
 * slots (rounded up to 256 bytes), then one int2 per row.
 * Verify index attention: candidate lists of topk keys for (ntiles + 255)
 * slots of 8 rows (rounded up to 256 bytes), a block-maximum scratch of
 * 256 x 8 x max_blocks fp32 (rounded up likewise), then one int2 per row.
 * Neither needs zeroing: every call writes what it reads.
 * Attention: 0 (its split-K partials are merged on chip); its ws arguments
 * are accepted and ignored.
 */
size_t m3s_workspace_bytes(int op, int32_t R, int32_t B, int32_t max_blocks, int32_t Hq,
                           int32_t Hkv, int32_t Hi, int32_t topk, int32_t max_q);

/*
 * Quantise-store. "[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache"
 * (ROCm/ATOM #2744), Design / Write path: the step's BF16 rows are quantised
 * into the paged planes at their real slots; per 16 elements
 * scale = e4m3(amax / 6) (saturating at 448), codes rounded half-to-even on the
 * e2m1 grid and saturating at 6. A group whose scale rounds to 0 stores zero
 * codes; a code's sign bit is the sign bit of the input.
 * Into an MXFP4 plane (dst.format == M3S_FMT_MXFP4; #2744, Follow-up: MXFP4
 * caches -- one E8M0 scale per 32 elements), per 32 elements the shared
 * exponent is E = floor(log2(amax)) - 2 clamped to [-127, 127] (amax 0 gives
 * -127; the pages name the format, this is its OCP MX rule), the scale byte
 * is E + 127, and each code is |x| / 2^E rounded half-to-even on the e2m1
 * grid, saturating at 6, with the sign bit of the input.
 *
 *   src          : BF16 [T][H][128] (row r, head h at src + r*src_row_stride + h*128)
 *   src_row_stride: elements between consecutive rows (>= H*128, multiple of 8)
 *   slot_mapping : int64 [T]; slot < 0 = pad row, skipped and its bytes untouched
 *                  ("NVFP4 sparse KV", Tests: pad rows stay unwritten)
 *   dst          : the plane pair; dst.num_heads must equal H
 * A slot >= dst.num_pages*128 sets M3S_DEVERR_SLOT and the row is skipped.
 * T == 0 is a no-op.
 */
int m3s_nvfp4_store(const uint16_t* src, int64_t src_row_stride, int32_t T, int32_t H,
                    const int64_t* slot_mapping, m3s_fp4_plane dst, int32_t* err,
                    void* stream);

/*
 * Batched quantise-store: up to M3S_MAX_STORE_JOBS tensors whose rows share
 * one slot mapping (a step's new K, V and index-K rows), in one launch. Each
 * job is quantised exactly as m3s_nvfp4_store would. `jobs` is a HOST array
 * (read during the call); each job's src row r holds job.H heads.
 */
#define M3S_MAX_STORE_JOBS 4
typedef struct {
  const uint16_t* src;    /* BF16 [T][H][128] device rows */
  int64_t src_row_stride; /* elements between rows (>= H*128, multiple of 8) */
  int32_t H;              /* heads per row; must equal dst.num_heads */
  m3s_fp4_plane dst;      /* either format; jobs may differ */
} m3s_store_job;

int m3s_nvfp4_store_batch(const m3s_store_job* jobs, int32_t njobs, int32_t T,
                          const int64_t* slot_mapping, int32_t* err, void* stream);

/*
 * m3s_nvfp4_store_batch and m3s_decode_rows in one launch: the step's writes
 * and its row map (#2744, Design / Attention: the row map is computed on
 * device; #2746, Summary: the step's K/V rows are quantised into the pages).
 * The store arguments as for m3s_nvfp4_store_batch (T == 0 or njobs == 0:
 * the row map alone), the row-map arguments and outputs as for
 * m3s_decode_rows (R == 0: the store alone). Same results as the two calls.
 */
int m3s_nvfp4_store_batch_rows(const m3s_store_job* jobs, int32_t njobs, int32_t T,
                               const int64_t* slot_mapping, const int32_t* cu_q, const int32_t* seq_len,
                               int32_t B, int32_t R, int32_t* row_req, int32_t* row_len, int32_t* err,
                               void* stream);

/*
 * Quantise-at-write. #2744, Follow-up: MXFP4 caches -- the quantisation moves
 * into the kernel that normalises and rotates the step's rows and writes the
 * cache, so there is no BF16 staging buffer and no separate store launch (the
 * unfused path, #2744 Summary / Write: the rows go BF16 to a staging buffer,
 * then the store quantises them). The normalisation and rotation belong to the
 * model; this call takes their parameters. Per job, for each row t and head h
 * of src (BF16 [T][H][128], row stride src_row_stride):
 *   RMSNorm, when norm_weight (fp32 [128]) is given:
 *     r = 1 / sqrt(sum_i(x_i^2) / 128 + eps), y_i = (x_i * r) * norm_weight[i];
 *     else y = x;
 *   RoPE, when job.rope != 0 (rotate-half on the first rotary_dim dims; c, s =
 *     rope_cos[t][i], rope_sin[t][i], fp32 [T][rotary_dim / 2]):
 *     o_i = y_i c - y_{i+rd/2} s,  o_{i+rd/2} = y_{i+rd/2} c + y_i s  (i < rd/2);
 *   the result rounded to BF16 (nearest, ties to even) -- the value the staging
 *   buffer would hold -- and then either quantised into dst at slot_mapping[t]
 *   exactly as m3s_nvfp4_store does (either format; pad rows skipped, a slot
 *   past the plane sets M3S_DEVERR_SLOT), or, when out is given, written to out
 *   as BF16 rows (queries: every row t).
 * Arithmetic: float32, each operation rounded on its own (no fused
 * multiply-add); the sum of squares in a fixed order (32 lanes each add the
 * squares of 4 consecutive elements left to right, then an xor butterfly over
 * offsets 16, 8, 4, 2, 1, lane 0's value taken), so the bytes are reproducible.
 * rotary_dim: a multiple of 8 in [8, 128] when any job rotates (else ignored);
 * rope_cos / rope_sin and norm weights 16-byte aligned; out_row_stride >= H*128
 * and a multiple of 8. T == 0 is a no-op.
 */
#define M3S_MAX_WRITE_JOBS 6
typedef struct {
  const uint16_t* src;      /* BF16 [T][H][128] device rows */
  int64_t src_row_stride;   /* elements between rows (>= H*128, multiple of 8) */
  int32_t H;                /* heads per row */
  const float* norm_weight; /* fp32 [128] RMSNorm weight, or NULL (no normalisation) */
  int32_t rope;             /* nonzero: rotate */
  m3s_fp4_plane dst;        /* destination plane (num_heads == H) when out is NULL */
  uint16_t* out;            /* BF16 [T][H][128] output rows, or NULL */
  int64_t out_row_stride;   /* elements between output rows */
} m3s_write_job;

int m3s_qk_norm_rope_store(const m3s_write_job* jobs, int32_t njobs, int32_t T,
                           const int64_t* slot_mapping, const float* rope_cos,
                           const float* rope_sin, int32_t rotary_dim, float eps, int32_t* err,
                           void* stream);

/*
 * Row map. #2744, Design / Attention: one launch maps each row to its request
 * and causal length, on device, so it is valid under CUDA-graph capture.
 * Request b owns rows cu_q[b] .. cu_q[b+1]-1 (Q_b rows) and holds seq_len[b]
 * tokens including them; its row j attends to seq_len[b] - Q_b + j + 1 tokens.
 * Rows r >= cu_q[B] are padding and get (row_req, row_len) = (-1, 0).
 *   cu_q int32 [B+1] (non-decreasing, cu_q[0] = 0), seq_len int32 [B],
 *   row_req, row_len int32 [R] outputs. B == 0 makes every row padding.
 */
int m3s_decode_rows(const int32_t* cu_q, const int32_t* seq_len, int32_t B, int32_t R,
                    int32_t* row_req, int32_t* row_len, void* stream);

/*
 * Lightning-indexer scoring with block top-k. #2744, Design / Index and Decode
 * score grid; "NVFP4 sparse KV", Summary (fused verify top-k emits ids only).
 * For row r of request b = row_req[r] with causal length L = row_len[r]:
 *   score[t] = sum_h w[r,h] * ReLU(q_idx[r,h,:] . k_hat[t,:]),  t < L,
 *   k_hat = the dequantised index key (index plane, one head; NVFP4, or MXFP4
 *           (exact when a key's four E8M0 scales lie within a factor 2^23 of
 *           each other; smaller groups beyond that are rounded in fp16)),
 *   block_score[blk] = max of score over the block's causal tokens,
 *   topk_ids[r] = the topk blocks with the highest block score, the lower id
 *                 on equal scores, sorted ascending, padded with -1.
 * Forced blocks (#2744's review of the fused verify top-k; "MXFP4 KV cache
 * for MiniMax-M3.1 on gfx950" (vllm #64198), Design: the init / local
 * sentinels): the first init_blocks and the last local_blocks blocks of each
 * row rank above every scored block, init above local; init blocks lower id
 * first, local blocks most recent first (so init + local > topk keeps the
 * row's newest blocks, its current token's block among them). 0, 0 = none;
 * negative counts are M3S_ERR_INVALID.
 *   q_idx BF16 [R][Hi][128], w fp32 [R][Hi], Hi <= 16,
 *   idx_k.num_heads == 1, block_table int32 [B][bt_stride] (logical block ->
 *   physical page), row_req / row_len from m3s_decode_rows,
 *   topk_ids int32 [R][topk] (topk <= 64),
 *   block_scores fp32 [R][bt_stride] or NULL: when given, also receives every
 *   row's block scores (entries past the row's block count are left as is).
 * Rows with row_req < 0 or row_len <= 0 produce -1 ids. Needs
 * ws_bytes >= m3s_workspace_bytes(M3S_OP_INDEX_SCORE_TOPK, ...) (for up to 256
 * rows none when block_scores is given: the scores go there), zeroed before
 * its first use when R > 256 (see there).
 * Two forms, by the number of rows. Above 256 rows (more than the scorer runs
 * CTAs) the top-k streams inside the scorer (#2744, Fused verify top-k: a
 * streaming top-k per chunk, then a merge): each warp keeps a running top-k as
 * it scores, each CTA leaves its share of a row as topk candidate keys in the
 * workspace, and the CTA that scores a row's last block merges the row's
 * candidates into its ids; one launch, no block-score matrix. Up to 256 rows
 * every row ends with the launch and those merges would form its tail: the
 * scorer writes the block scores and a second launch selects.
 */
int m3s_index_score_topk(const uint16_t* q_idx, const float* w, int32_t Hi,
                         m3s_fp4_plane idx_k, const int32_t* block_table, int32_t bt_stride,
                         const int32_t* row_req, const int32_t* row_len, int32_t R, int32_t B,
                         int32_t topk, int32_t init_blocks, int32_t local_blocks,
                         int32_t* topk_ids, float* block_scores, void* ws, size_t ws_bytes,
                         int32_t* err, void* stream);

/*
 * The two halves of m3s_index_score_topk, for callers that want the block
 * scores alone or time the scorer by itself.
 * m3s_index_block_scores: block_scores fp32 [R][bs_stride] (bs_stride >=
 * bt_stride) receives, for every valid row, the block score of each of its
 * ceil(row_len/128) blocks; other entries are left as is.
 * m3s_block_topk: topk_ids [R][topk] from those scores (ties to the lower id,
 * ascending, -1 padded, forced blocks as above); row_req may be NULL (then
 * rows are taken as valid when 0 < row_len <= bt_stride*128 and B > 0).
 */
int m3s_index_block_scores(const uint16_t* q_idx, const float* w, int32_t Hi,
                           m3s_fp4_plane idx_k, const int32_t* block_table, int32_t bt_stride,
                           const int32_t* row_req, const int32_t* row_len, int32_t R, int32_t B,
                           float* block_scores, int32_t bs_stride, int32_t* err, void* stream);
int m3s_block_topk(const float* block_scores, int32_t bs_stride, const int32_t* row_req,
                   const int32_t* row_len, int32_t R, int32_t B, int32_t bt_stride, int32_t topk,
                   int32_t init_blocks, int32_t local_blocks, int32_t* topk_ids, void* stream);

/*
 * Indexer context parallelism. #2744, review thread on the unused page-16
 * tables: with indexer CP one request's index keys are split over ranks; each
 * rank scores its share and the ranks' candidate keys are merged
 * (merge_candidate_keys) into the top-k. (The pages' engine refuses CP
 * together with the FP4 index at startup; this library does not.)
 *
 * Candidate keys, uint64, larger = better, 0 = an empty slot:
 *   a scored block:  high word = the fp32 block score's order-preserving bits
 *                    (x >= 0: bits | 0x80000000, x < 0: ~bits, -0 as +0),
 *                    low word = 0xFFFFFFFF - block id (ties to the lower id);
 *   a forced init block:  0xFFFFFFFF : 0xFFFFFFFF - id;
 *   a forced local block: 0xFFFFFFFE : id.
 *
 * m3s_index_score_candidates: the rows' top-k over a slice of each request's
 * blocks, as candidate keys cand_keys uint64 [R][topk] (descending, 0-padded),
 * with the request's block ids and token positions: request b's slice holds
 * its blocks blk_begin[b] .. blk_begin[b] + blk_count[b] - 1 (int32 [B],
 * device), local block j at block_table[b][j] of this slice's table; row r
 * (length row_len[r], the whole request's causal length) scores the slice's
 * tokens below row_len[r]. Forced blocks are placed by the row's own block
 * count. Other arguments as for m3s_index_score_topk. One launch (the
 * streaming form); ws_bytes >= m3s_workspace_bytes(M3S_OP_INDEX_CANDIDATES,
 * ...), zeroed before its first use (every call leaves it zeroed).
 *
 * m3s_merge_candidates: the top-k ids of each row from n_lists ranks' candidate
 * keys (cand_keys uint64 [n_lists][R][topk], each row's list descending),
 * ascending and -1 padded, as m3s_index_score_topk returns them; n_lists <= 256.
 * Merging every slice's candidates gives the unsplit call's ids: each block of
 * a row's top-k is among its own slice's top-k.
 */
int m3s_index_score_candidates(const uint16_t* q_idx, const float* w, int32_t Hi, m3s_fp4_plane idx_k,
                               const int32_t* block_table, int32_t bt_stride, const int32_t* blk_begin,
                               const int32_t* blk_count, const int32_t* row_req, const int32_t* row_len,
                               int32_t R, int32_t B, int32_t topk, int32_t init_blocks,
                               int32_t local_blocks, uint64_t* cand_keys, void* ws, size_t ws_bytes,
                               int32_t* err, void* stream);
int m3s_merge_candidates(const uint64_t* cand_keys, int32_t n_lists, int32_t R, int32_t topk,
                         int32_t* topk_ids, void* stream);

/*
 * m3s_index_score_topk without a caller workspace. The pages have no
 * counterpart to this call; it is an integration variant of
 * m3s_index_score_topk (same arguments minus block_scores / ws / ws_bytes and
 * without forced blocks, the same result as that call with init_blocks =
 * local_blocks = 0) for callers that cannot allocate device memory at call time:
 * a C host that links only this library and owns no device allocator, or an
 * engine plugin whose device memory is budgeted once at start-up.
 * The block-score scratch is a file-scope device array of
 * M3S_STATIC_SCRATCH_BYTES (4 MiB), one per device; the call allocates
 * nothing. Limits, checked before any launch: R above 8192 returns
 * M3S_ERR_UNSUPPORTED (as for m3s_index_score_topk); R * max(bt_stride, 1) * 4
 * bytes above the scratch size returns M3S_ERR_WORKSPACE. Every call looks the
 * array's address up in the current context (cudaGetSymbolAddress); the first
 * call on a device also loads the library's device module and should come
 * before any stream capture. Nothing in the scratch needs to start at zero.
 * Every call on a device shares the one scratch: calls that overlap on the GPU
 * (e.g. on two unordered streams) race and may return wrong ids.
 */
#define M3S_STATIC_SCRATCH_BYTES (4u << 20)
int m3s_index_score_topk_static(const uint16_t* q_idx, const float* w, int32_t Hi,
                                m3s_fp4_plane idx_k, const int32_t* block_table,
                                int32_t bt_stride, const int32_t* row_req, const int32_t* row_len,
                                int32_t R, int32_t B, int32_t topk, int32_t* topk_ids,
                                int32_t* err, void* stream);

/*
 * Fused verify score + top-k. #2744, Design / Fused verify top-k: for
 * speculative-verify rows, index scoring and top-k in one pass over each
 * request's keys, emitting top-k ids only (all the sparse attention reads).
 * Same result as m3s_index_score_topk on the same rows; here the rows of one
 * request are scored together (their queries share every key read), which
 * also serves a prefill chunk (one request, many rows).
 *   cu_q int32 [B+1] groups rows by request (as for m3s_decode_rows),
 *   row_len int32 [R] their causal lengths (m3s_decode_rows),
 *   max_q >= every cu_q[b+1]-cu_q[b] (sizes the request-row tiling).
 * Other arguments as for m3s_index_score_topk (the index plane NVFP4 or MXFP4,
 * with the same exactness); rows past cu_q[B] get -1 ids. As for
 * m3s_index_score_topk, more than 256 tiles stream the top-k inside the scorer
 * (one launch; the epilogue leaves each row's block maxima in a per-CTA score
 * scratch, one warp a row selects at its segment's end), else block scores and
 * a second launch. Needs ws_bytes >= m3s_workspace_bytes(M3S_OP_VERIFY_SCORE_TOPK,
 * ...), zeroed before its first use in the streaming form.
 */
int m3s_verify_score_topk(const uint16_t* q_idx, const float* w, int32_t Hi,
                          m3s_fp4_plane idx_k, const int32_t* block_table, int32_t bt_stride,
                          const int32_t* cu_q, const int32_t* row_len, int32_t B, int32_t R,
                          int32_t max_q, int32_t topk, int32_t init_blocks, int32_t local_blocks,
                          int32_t* topk_ids, void* ws, size_t ws_bytes, int32_t* err,
                          void* stream);

/*
 * Decode rows end to end: index scoring, top-k and block-sparse attention in
 * two launches. #2744, Design / Index and Design / Attention: the indexer's
 * top-k block ids of each row address the blocks the row attends over. The
 * scorer leaves, for every row, each of its CTAs' top-k candidate keys over the
 * blocks it scored (the key order of m3s_index_score_topk: score, ties to the
 * lower id, forced blocks first); the attention merges a row's candidates
 * before it reads the row's pages. topk_ids, out and lse are what
 * m3s_index_score_topk followed by m3s_sparse_attention return (same ids, and
 * the attention then computes the same sums in the same order).
 * Arguments as for those two calls; topk_ids int32 [R][topk] is written.
 * ws_bytes >= m3s_workspace_bytes(M3S_OP_INDEX_ATTENTION, ...) (no zeroing
 * needed: every call writes what it reads). R <= 8192.
 */
int m3s_index_attention(const uint16_t* q_idx, const float* w, int32_t Hi, m3s_fp4_plane idx_k,
                        const uint16_t* q, int32_t Hq, int32_t Hkv, m3s_fp4_plane k, m3s_fp4_plane v,
                        const int32_t* block_table, int32_t bt_stride, int32_t B, const int32_t* row_req,
                        const int32_t* row_len, int32_t R, int32_t topk, int32_t init_blocks,
                        int32_t local_blocks, float sm_scale, int32_t* topk_ids, uint16_t* out, float* lse,
                        void* ws, size_t ws_bytes, int32_t* err, void* stream);

/*
 * Verify rows end to end: the fused verify scoring, top-k and block-sparse
 * attention in two launches. #2744, Fused verify top-k (a request's rows scored
 * together against each block, the top-k kept per chunk and merged) and
 * Design / Attention. The verify scorer (tiles of up to 8 rows of one request,
 * as m3s_verify_score_topk) leaves, for every row, each of its CTAs' top-k
 * candidate keys over the blocks it scored; the attention merges a row's
 * candidates before it reads the row's pages. topk_ids, out and lse are what
 * m3s_verify_score_topk followed by m3s_sparse_attention return.
 * Arguments: those of m3s_verify_score_topk (cu_q int32 [B + 1], row_len,
 * max_q) and of m3s_sparse_attention (q, heads, K / V planes, row_req int32
 * [R], the row map of the same rows). ws_bytes >=
 * m3s_workspace_bytes(M3S_OP_VERIFY_INDEX_ATTENTION, R, B, bt_stride, Hq, Hkv,
 * Hi, topk, max_q) (no zeroing needed). B * ceil(max_q / 8) <= 8192 tiles, else
 * M3S_ERR_UNSUPPORTED. Rows at or past cu_q[B] (all of them when B = 0) get
 * no ids (-1), zero output and lse -inf; topk = 0 launches only the attention,
 * which gives every row that result.
 */
int m3s_verify_index_attention(const uint16_t* q_idx, const float* w, int32_t Hi, m3s_fp4_plane idx_k,
                               const uint16_t* q, int32_t Hq, int32_t Hkv, m3s_fp4_plane k, m3s_fp4_plane v,
                               const int32_t* block_table, int32_t bt_stride, int32_t B, const int32_t* cu_q,
                               const int32_t* row_req, const int32_t* row_len, int32_t R, int32_t max_q,
                               int32_t topk, int32_t init_blocks, int32_t local_blocks, float sm_scale,
                               int32_t* topk_ids, uint16_t* out, float* lse, void* ws, size_t ws_bytes,
                               int32_t* err, void* stream);

/*
 * Block-sparse attention over the selected NVFP4 pages. "NVFP4 sparse KV",
 * Summary / Attention and #2744 Design / Attention: decode and prefill rows
 * attend over their top-k blocks, addressed by the top-k block ids and the
 * request block table, against the dequantised K/V.
 * For row r (request b = row_req[r], causal length L = row_len[r]) and q head h
 * (KV head h / (Hq/Hkv)), over the tokens t of the listed blocks with t < L:
 *   out[r,h] = sum_t softmax_t(sm_scale * q[r,h] . k_hat[t]) v_hat[t],
 *   lse[r,h] = log sum_t exp(sm_scale * q[r,h] . k_hat[t])   (natural log).
 *   q BF16 [R][Hq][128], out BF16 [R][Hq][128], lse fp32 [R][Hq] or NULL,
 *   k / v planes with num_heads == Hkv, topk_ids int32 [R][topk] LOGICAL
 *   block ids within the request (-1 = skip). Hq/Hkv <= 16, topk <= 64,
 *   block_table int32 [B][bt_stride]; a row with row_req outside [0, B) or a
 *   length beyond the table sets M3S_DEVERR_ROW and outputs zeros.
 * An id >= the row's block count (or >= bt_stride) sets M3S_DEVERR_BLOCK_ID
 * and is skipped (never wrapped onto another page). A row with no token
 * (pad row, all ids -1) outputs zeros and lse = -inf. Duplicate ids count
 * their block once per occurrence.
 * k and v share one format (NVFP4 or MXFP4; mixed formats return
 * M3S_ERR_UNSUPPORTED, as the pages' startup refuses mixing them: #2744,
 * Follow-up: MXFP4 caches). The products are fp16 x fp16 (q is scaled per head
 * into f16's range, see the conventions above): NVFP4 K/V dequantise exactly
 * to fp16; MXFP4 K is scaled
 * per token by its largest exponent and V per 32-dim group by the largest
 * exponent of the row's selected tokens so far, the factors re-applied in
 * fp32, which is exact while the exponents so normalised span at most 23.
 */
int m3s_sparse_attention(const uint16_t* q, int32_t Hq, int32_t Hkv, m3s_fp4_plane k,
                         m3s_fp4_plane v, const int32_t* block_table, int32_t bt_stride,
                         int32_t B, const int32_t* row_req, const int32_t* row_len, const int32_t* topk_ids,
                         int32_t topk, int32_t R, float sm_scale, uint16_t* out, float* lse,
                         void* ws, size_t ws_bytes, int32_t* err, void* stream);

/* Library version string (static storage). */
const char* m3s_version(void);

#ifdef __cplusplus
}
#endif

#endif /* M3S_H_ */
