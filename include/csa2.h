/*
 * csa2.h - C ABI of the CSA2 decode path over an FP4 global KV cache (sm_103a).
 *
 * The method is DeepSeek-V4.1-Flash's Compressed Sparse Attention 2 as the
 * pages describe it:
 *   - origotech.dev, "DeepSeek V4.1-Flash 내부: KV 캐시, 1017 업데이트, Harness
 *     스택", section "아키텍처는 어떻게 KV 캐시를 줄이나", subsections
 *     "Compressed Sparse Attention 2(CSA2)" (Full / Reindex / Reuse modes, the
 *     decoder's layer pattern, top-k 512, 128-token window, 2,048 blocks of 8
 *     kept by the first Full layer) and "FP4와 SWA Bounded Replay" (main KV in
 *     FP4 E2M1 with one E4M3 scale per 16 channels, quantised after RoPE; SWA
 *     KV in FP8);
 *   - trawling.dev, "DeepSeek-V4.1-Flash 공개 ...", section "CSA2와 FP4 KV
 *     캐싱" (the same modes and format; the hierarchical indexer bounds the
 *     deep layers' indexer cost independently of context length);
 *   - ttj.kr, "DeepSeek-V4.1-Flash, KV 캐시를 토큰당 890바이트까지 압축하다",
 *     section "CSA2와 어텐션 재설계" (local window plus global sparse retrieval).
 * Dimensions the pages leave open are fixed here: main KV is MQA with 128
 * channels used as both K and V, channels 64..127 rotated; the indexer has 8
 * query heads of dim 64 against one FP8 key per token with a float32 scale,
 * and scores sigma_t = s_t * sum_h w_h * max(q_h . k_t, 0).
 *
 * Conventions for every entry point:
 *   - all buffers are caller-owned device memory unless stated otherwise;
 *     the library allocates nothing.  Between calls it keeps only (a) a table
 *     of per-device launch facts (SM count, CTAs per SM of a kernel, the
 *     opt-in to large dynamic shared memory), filled on a device's first call
 *     and keyed by device, so that several host threads and several devices
 *     can call concurrently, and (b) the static scratch array of
 *     indexer_reindex_select_static (see its Set-up and Sharing notes);
 *   - every call only enqueues work on `stream` (no synchronisation, no
 *     host<->device copy), so calls can be captured into CUDA graphs;
 *   - the return value is a CSA2_STATUS code; arguments are validated on the
 *     host before anything is launched (null pointers, sizes out of range,
 *     misaligned buffers -> CSA2_ERR_INVALID_ARG, nothing enqueued);
 *   - problems only visible on the device (an out-of-range sequence id,
 *     position, length or index) make the kernel skip the offending item and
 *     OR a CSA2_DEVERR_* bit into *d_err (a caller-owned device int32 that the
 *     caller zeroes and reads back after synchronising).  d_err may not be NULL;
 *   - bf16 arguments are passed as their 16-bit patterns (uint16_t).
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *csa2_stream_t; /* identical to cudaStream_t */
typedef struct CUevent_st *csa2_event_t;   /* identical to cudaEvent_t  */

enum csa2_status {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,    /* bad pointer, size or alignment; nothing launched        */
  CSA2_ERR_WORKSPACE = 2,      /* workspace pointer null/misaligned or smaller than needed */
  CSA2_ERR_UNSUPPORTED = 3,    /* current device is not compute capability 10.3           */
  CSA2_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed                    */
  CSA2_ERR_DEVICE_TIMEOUT = 5  /* reserved: a bounded device-side wait gave up            */
};

enum csa2_device_error_bits {
  CSA2_DEVERR_SEQ = 1,     /* sequence id outside [0, B)                               */
  CSA2_DEVERR_POS = 2,     /* position < 0, >= rope_len, or cache row outside [0,T_cap) */
  CSA2_DEVERR_LEN = 4,     /* seq_len < 0, > max_len, or seq_base+seq_len > T_cap      */
  CSA2_DEVERR_INDEX = 8,   /* a top-k index beyond the query position or the cache     */
  CSA2_DEVERR_POOL = 16,   /* a pool block id outside the sequence                     */
  CSA2_DEVERR_TIMEOUT = 32 /* a bounded wait gave up                                   */
};

#define CSA2_D 128        /* main KV channels (K = V)                */
#define CSA2_D_ROPE 64    /* rotated channels: 64..127               */
#define CSA2_D_IDX 64     /* indexer key / query dim                 */
#define CSA2_H_IDX 8      /* indexer query heads                     */
#define CSA2_MAX_B 1024   /* sequences per call                      */
#define CSA2_MAX_SWA_LAYERS 32

/*
 * One global cache shared by every decoder layer (main KV + indexer key) for
 * B sequences.  Sequence b's position p lives in row seq_base[b] + p.
 * Layout in HBM (row-major, no padding):
 *   kv_codes  [T_cap][64]  uint8  two E2M1 codes per byte: channel 2j in bits
 *                                  0-3, channel 2j+1 in bits 4-7 (bit 3 of a
 *                                  nibble is the sign)
 *   kv_scales [T_cap][8]   uint8  E4M3 scale of channels 16g..16g+15
 *   ik_codes  [T_cap][64]  uint8  E4M3 indexer key
 *   ik_scale  [T_cap]      float  per-token indexer key scale
 * seq_base and seq_len are device arrays of B entries; seq_len[b] is the
 * number of valid positions (rows seq_base[b] .. seq_base[b]+seq_len[b]-1).
 * All four data arrays must be 16-byte aligned.
 */
typedef struct csa2_cache {
  uint8_t *kv_codes;
  uint8_t *kv_scales;
  uint8_t *ik_codes;
  float *ik_scale;
  const int64_t *seq_base;
  const int32_t *seq_len;
  int32_t B;
  int64_t T_cap;
} csa2_cache;

/*
 * One decoder layer's sliding-window KV in FP8: a ring of `ring` slots per
 * sequence; position p lives in slot p % ring.
 *   codes [B][ring][128] uint8 E4M3 (RoPE applied before quantisation)
 *   scale [B][ring]      float per-token scale
 */
typedef struct csa2_swa {
  uint8_t *codes;
  float *scale;
  int32_t ring;
} csa2_swa;

/* Optional timing hook: when non-NULL, the call records `start` just before
 * and `stop` just after its dominant kernel (the indexer scan), on `stream`. */
typedef struct csa2_profile {
  csa2_event_t start;
  csa2_event_t stop;
} csa2_profile;

enum csa2_op {
  CSA2_OP_FULL_SELECT = 1,
  CSA2_OP_REINDEX_SELECT = 2,
  CSA2_OP_ATTN_DECODE = 3,
  CSA2_OP_VERIFY_SELECT = 4,
  CSA2_OP_CHUNKED_SELECT = 5
};

/* Human-readable name of a status code (static string). */
const char *csa2_status_string(int status);

/*
 * Workspace bytes needed by one call of `op` (written to *bytes).
 *   FULL_SELECT / REINDEX_SELECT: B, max_len, block, n_keep_blocks, topk used.
 *   ATTN_DECODE: T (query rows), H (heads), topk, window used.
 *   VERIFY_SELECT: T (query rows), block, n_keep_blocks, topk used.
 *   CHUNKED_SELECT: T (query rows), max_len, block, n_keep_blocks, topk used.
 * Returns CSA2_ERR_INVALID_ARG for out-of-range sizes.  Workspace must be
 * 256-byte aligned; its contents need not be initialised and are clobbered.
 */
int csa2_workspace_bytes(int op, int32_t B, int64_t max_len, int32_t block, int32_t n_keep_blocks,
                         int32_t topk, int64_t T, int32_t H, int32_t window, size_t *bytes);

/*
 * kv_append_fp4 - RoPE, then quantise-and-append n new tokens.
 * (origotech.dev deep dive, subsection "FP4와 SWA Bounded Replay")
 *   cache          the shared global cache (written: rows seq_base[seq_id[i]] + pos[i])
 *   swa_layers     host array of n_swa_layers ring descriptors (may be NULL if 0)
 *   kv_new         bf16 [n][128] main KV before RoPE
 *   ik_new         bf16 [n][64] indexer key, or NULL to leave the indexer rows untouched
 *   swa_new        bf16 [n_swa_layers][n][128] per-layer window KV before RoPE, or NULL
 *   rope_cos/sin   float [rope_len][32]: angle of pair i (channels 64+2i, 65+2i)
 *                  at position p is read from row p
 *   seq_id, pos    int32 [n], int64 [n]
 * Per token: channels 64..127 rotated in float32 (r0 = x0*c - x1*s,
 * r1 = x0*s + x1*c, each product and sum rounded separately); each 16-channel
 * group gets s = E4M3(amax/6) (round to nearest even, saturating) and E2M1
 * codes of |r|/s (nearest, ties to even, saturating at 6) with r's sign bit;
 * the indexer key gets s = amax/448 and E4M3(x/s); each SWA layer's vector is
 * rotated like the main KV and quantised like the indexer key into slot
 * pos % ring.  n may be 0.  Tokens with a bad seq_id or position are skipped
 * (CSA2_DEVERR_SEQ / _POS).  Requires n_swa_layers <= CSA2_MAX_SWA_LAYERS.
 */
int kv_append_fp4(const csa2_cache *cache, const csa2_swa *swa_layers, int32_t n_swa_layers,
                  const uint16_t *kv_new, const uint16_t *ik_new, const uint16_t *swa_new,
                  const float *rope_cos, const float *rope_sin, int64_t rope_len,
                  const int32_t *seq_id, const int64_t *pos, int64_t n, int32_t *d_err,
                  csa2_stream_t stream);

/*
 * swa_refill_fp8 - rebuild the sliding-window rings of every layer from replayed
 * window KV, leaving the global cache untouched.
 * (origotech.dev deep dive, subsection "FP4와 SWA Bounded Replay": the FP8 window
 * KV is not persisted; after a restart the last window of tokens is replayed and
 * its per-layer KV re-appended)
 *   swa_layers     host array of n_swa_layers (1..CSA2_MAX_SWA_LAYERS) ring descriptors
 *   B              number of sequences (seq_id must lie in [0, B))
 *   swa_new        bf16 [n_swa_layers][n][128] replayed window KV before RoPE
 *   rope_cos/sin, seq_id, pos, n, d_err: as kv_append_fp4
 * Each token's vector of each layer is rotated and quantised exactly as
 * kv_append_fp4 does for its SWA layers (same bytes) into slot pos % ring.
 * Tokens with a bad seq_id or position are skipped (CSA2_DEVERR_SEQ / _POS).
 */
int swa_refill_fp8(const csa2_swa *swa_layers, int32_t n_swa_layers, int32_t B, const uint16_t *swa_new,
                   const float *rope_cos, const float *rope_sin, int64_t rope_len, const int32_t *seq_id,
                   const int64_t *pos, int64_t n, int32_t *d_err, csa2_stream_t stream);

/*
 * indexer_full_select - a Full layer's indexer over every cached position.
 * (origotech.dev deep dive, subsection "Compressed Sparse Attention 2(CSA2)":
 * the first Full layer picks 2,048 blocks of 8 positions and its top-512)
 *   q_idx          bf16 [B][8][64] this layer's indexer queries
 *   w              float [B][8]    head weights (>= 0)
 *   block          positions per block: 1, 2, 4, 8 or 16 (default 8)
 *   n_keep_blocks  blocks kept in the pool, 1..4096 (default 2048)
 *   topk           positions selected, 1..min(1024, n_keep_blocks) (default 512)
 *   max_len        host upper bound on every seq_len[b] (sizes the workspace)
 *   pool_blocks    int32 [B][n_keep_blocks] out: the min(n_keep, ceil(L/block))
 *                  best blocks by (block score desc, id asc), ascending, -1 padded;
 *                  a block's score is the max of its members' scores
 *   topk_idx       int32 [B][topk] out: the min(topk, L) best positions by
 *                  (score desc, position asc), ascending, -1 padded
 * Ranking is exact: approximate tensor-core scores carry a rigorous error
 * bound, and every item whose bound straddles a selection threshold is
 * rescored exactly (64-bit integer dot products) before the final choice.
 */
int indexer_full_select(const csa2_cache *cache, const uint16_t *q_idx, const float *w,
                        int32_t block, int32_t n_keep_blocks, int32_t topk, int64_t max_len,
                        int32_t *pool_blocks, int32_t *topk_idx, void *ws, size_t ws_bytes,
                        int32_t *d_err, const csa2_profile *prof, csa2_stream_t stream);

/*
 * indexer_reindex_select - a Reindex layer: rescore only the pool's positions
 * with this layer's indexer queries and the Full layer's keys, pick top-k.
 * (origotech.dev deep dive, subsection "Compressed Sparse Attention 2(CSA2)")
 *   pool_blocks    int32 [B][n_keep_blocks] from indexer_full_select (-1 entries ignored)
 *   topk_idx       int32 [B][topk] out, ascending, -1 padded
 * Other arguments as indexer_full_select.  A pool id beyond the sequence sets
 * CSA2_DEVERR_POOL and is ignored.  A Reuse layer needs no call: it passes
 * the same topk_idx buffer on.
 */
int indexer_reindex_select(const csa2_cache *cache, const uint16_t *q_idx, const float *w,
                           const int32_t *pool_blocks, int32_t block, int32_t n_keep_blocks,
                           int32_t topk, int64_t max_len, int32_t *topk_idx, void *ws,
                           size_t ws_bytes, int32_t *d_err, csa2_stream_t stream);

/*
 * indexer_reindex_select_static - indexer_reindex_select for callers that
 * cannot allocate device memory.  The paper has no counterpart: this is a
 * calling convention, not a step of the method.
 *
 * Some callers have no way to obtain a workspace: a plugin inside an engine
 * whose memory planner owns every byte of the device and forbids cudaMalloc,
 * or code on a latency-critical path where cudaMalloc/cudaFree would
 * synchronise the device.  This entry point takes the same arguments as
 * indexer_reindex_select minus ws/ws_bytes, gives the same result, and
 * allocates nothing: its scratch is one static device array of
 * CSA2_STATIC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits.
 *   Limit: the call needs 4*B*(8196 + n_keep_blocks*(1 + 6*block)) bytes of
 *   scratch (each of its 9 arrays rounded up to 256 bytes); every call with
 *   B*n_keep_blocks*block <= 524,288 and B <= 64 fits.  A larger call returns CSA2_ERR_WORKSPACE and
 *   launches nothing.
 *   Set-up: the first call on each device resolves the array's device address
 *   with that device current; make that first call before any stream capture.
 *   Sharing: every call uses the same array and leaves its contents behind
 *   (the call clears what must start at zero).  Calls whose kernels overlap
 *   on the GPU (different streams, or several host threads) race on it:
 *   serialise them, for example on one stream.
 * Status codes, device error bits and output layout are indexer_reindex_select's.
 */
#define CSA2_STATIC_SCRATCH_BYTES (16u << 20)
int indexer_reindex_select_static(const csa2_cache *cache, const uint16_t *q_idx, const float *w,
                                  const int32_t *pool_blocks, int32_t block, int32_t n_keep_blocks,
                                  int32_t topk, int64_t max_len, int32_t *topk_idx, int32_t *d_err,
                                  csa2_stream_t stream);

/*
 * indexer_chunked_select - the Full layer's selection for many query rows at once, each
 * over its session's positions up to its own (a chunk of prefill queries).
 * (origotech.dev deep dive, subsection "Compressed Sparse Attention 2(CSA2)": a Full
 * layer scores every cached position with its own indexer queries and keeps 2,048 blocks
 * of 8 plus the top-512 positions; a query sees the positions up to its own)
 *   q_idx          bf16 [T][8][64], w float [T][8]: each row's indexer queries and weights
 *   q_seq, q_pos   int32 [T], int64 [T]: session and position of each row
 *   T              rows, 0..2^24
 *   max_len        >= q_pos[r] + 1 for every row (bounds the workspace)
 *   pool_blocks    int32 [T][n_keep_blocks] out, topk_idx int32 [T][topk] out: for row r,
 *                  exactly what indexer_full_select returns for a session made of the
 *                  first q_pos[r] + 1 positions of session q_seq[r]
 *   ws/ws_bytes    csa2_workspace_bytes(CSA2_OP_CHUNKED_SELECT, ...)
 * Rows are processed in groups of CSA2_MAX_B.  A row with a bad q_seq or q_pos selects
 * nothing (all -1) and sets CSA2_DEVERR_SEQ / _POS.
 */
int indexer_chunked_select(const csa2_cache *cache, const uint16_t *q_idx, const float *w, const int32_t *q_seq,
                           const int64_t *q_pos, int64_t T, int32_t block, int32_t n_keep_blocks, int32_t topk,
                           int64_t max_len, int32_t *pool_blocks, int32_t *topk_idx, void *ws, size_t ws_bytes,
                           int32_t *d_err, csa2_stream_t stream);

/*
 * indexer_verify_select - the Reindex selection for several query rows per session,
 * each with its own indexer queries and a causal limit: the rows verifying a batch
 * of drafted positions in speculative decoding.
 * (origotech.dev deep dive, section "아키텍처는 어떻게 KV 캐시를 줄이나", the DSpark
 * item of the remaining stack: a drafter proposes 5 positions at once, which are then
 * verified; the selection itself is the Reindex rule of subsection "Compressed Sparse
 * Attention 2(CSA2)")
 *   q_idx          bf16 [T][8][64] indexer queries of each row
 *   w              float [T][8]    head weights of each row
 *   q_seq, q_pos   int32 [T], int64 [T]: session and position of each row
 *   T              rows, 0..65535
 *   pool_blocks    int32 [B][n_keep_blocks] each session's pool (shared by its rows),
 *                  ascending, -1 entries ignored
 *   topk_idx       int32 [T][topk] out: the min(topk, candidates) best positions
 *                  p' <= q_pos[r] among the pool's positions, by (score desc,
 *                  position asc), ascending, -1 padded
 *   ws/ws_bytes    csa2_workspace_bytes(CSA2_OP_VERIFY_SELECT, ...)
 * Other arguments as indexer_reindex_select.  A row with a bad q_seq or q_pos
 * selects nothing and sets CSA2_DEVERR_SEQ / _POS; a pool id beyond its session's
 * length sets CSA2_DEVERR_POOL; pool positions after q_pos are not candidates.
 */
int indexer_verify_select(const csa2_cache *cache, const uint16_t *q_idx, const float *w, const int32_t *q_seq,
                          const int64_t *q_pos, int64_t T, const int32_t *pool_blocks, int32_t block,
                          int32_t n_keep_blocks, int32_t topk, int64_t max_len, int32_t *topk_idx, void *ws,
                          size_t ws_bytes, int32_t *d_err, csa2_stream_t stream);

/*
 * sparse_attn_decode - gathered FP4 dequantisation fused into sparse attention.
 * (ttj.kr article, section "CSA2와 어텐션 재설계"; origotech.dev deep dive,
 * subsection "Compressed Sparse Attention 2(CSA2)")
 *   swa            this layer's window ring (host struct)
 *   q              bf16 [T][H][128] (16-byte aligned); H a multiple of 16, <= 128
 *   q_seq, q_pos   int32 [T], int64 [T]: sequence and position of each query row
 *   topk_idx       int32 [T][topk] positions (<= q_pos), -1 entries skipped
 *   window         window length W (0..1024, <= swa->ring)
 *   softmax_scale  tau (use 1/sqrt(128))
 *   out            float [T][H][128] (16-byte aligned) = sum_j softmax(z)_j * v_j, z_j = tau * q . k_j
 *   lse            float [T][H] = log sum_j exp(z_j), or NULL
 * One softmax spans the valid selected rows (FP4, dequantised exactly) and
 * the window rows max(0, p-W+1)..p (FP8 value times the row's scale); V = K.
 * With no rows, out = 0 and lse = -inf.
 */
int sparse_attn_decode(const csa2_cache *cache, const csa2_swa *swa, const uint16_t *q, int32_t H,
                       int64_t T, const int32_t *q_seq, const int64_t *q_pos, const int32_t *topk_idx,
                       int32_t topk, int32_t window, float softmax_scale, float *out, float *lse,
                       void *ws, size_t ws_bytes, int32_t *d_err, csa2_stream_t stream);
/* (sparse_attn_decode needs no workspace: ws may be NULL and ws_bytes 0.) */

/* ---- test-only exports (same device code as the entry points above) ---- */

/* FP4 group quantiser of kv_append_fp4 on raw float32 groups (no RoPE):
 * x [n][16] -> codes [n][8] (packed as in kv_codes), scales [n]. */
int csa2_test_quantize_fp4(const float *x, int64_t n_groups, uint8_t *codes, uint8_t *scales,
                           csa2_stream_t stream);

/* Per-token FP8 quantiser of kv_append_fp4: x [n][C] (C = 64 or 128) ->
 * codes [n][C], scale [n]. */
int csa2_test_quantize_fp8(const float *x, int64_t n, int32_t C, uint8_t *codes, float *scale,
                           csa2_stream_t stream);

/* Approximate indexer scores of the scan (block 8) for every position of every
 * sequence: sigma [B][max_len] (entries at and beyond seq_len[b] untouched),
 * and bound [B+1] (device doubles): bound[b] = E_b and bound[B] = r, such that
 * |sigma_approx - sigma_exact| <= E_b + r * sigma_approx.  Workspace as for
 * CSA2_OP_FULL_SELECT with block 8 and n_keep_blocks 1. */
int csa2_test_index_scores(const csa2_cache *cache, const uint16_t *q_idx, const float *w,
                           int64_t max_len, float *sigma, double *bound, void *ws, size_t ws_bytes,
                           int32_t *d_err, csa2_stream_t stream);

/* Test: the tensor-core scores of T <= CSA2_MAX_B chunked-query rows (rows 16j..16j+15 must
 * share a session) into sigma [T][max_len] (device floats, positions > q_pos[r] untouched)
 * and bound [T+1] (device doubles) as for csa2_test_index_scores.  Workspace as for
 * CSA2_OP_CHUNKED_SELECT with block 8 and n_keep_blocks 1. */
int csa2_test_chunk_scores(const csa2_cache *cache, const uint16_t *q_idx, const float *w, const int32_t *q_seq,
                           const int64_t *q_pos, int64_t T, int64_t max_len, float *sigma, double *bound, void *ws,
                           size_t ws_bytes, int32_t *d_err, csa2_stream_t stream);

/* Test: the per-device launch-fact table with an explicit device id and no CUDA call.
 * Returns the value held for (device, site, key), or stores and returns `value` if there
 * is none (a negative value is returned without being stored). */
int csa2_test_device_memo(int device, int site, int64_t key, int value);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
