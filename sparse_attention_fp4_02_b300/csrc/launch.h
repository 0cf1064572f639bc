// Internal launchers of the CSA2 library (host side).
#pragma once

#include <cstddef>
#include <cstdint>
#include <functional>
#include <cuda_runtime.h>

#include "csa2.h"

namespace csa2 {

cudaError_t launch_append(const csa2_cache &c, const csa2_swa *swa, int n_swa, const uint16_t *kv_new,
                          const uint16_t *ik_new, const uint16_t *swa_new, const float *cos,
                          const float *sin, int64_t rope_len, const int32_t *seq_id, const int64_t *pos,
                          int64_t n, int32_t *d_err, cudaStream_t st);
cudaError_t launch_test_fp4(const float *x, int64_t n_groups, uint8_t *codes, uint8_t *scales,
                            cudaStream_t st);
cudaError_t launch_test_fp8(const float *x, int64_t n, int C, uint8_t *codes, float *scale, cudaStream_t st);

// ---- indexer ----
struct IndexerWs {           // carved out of the caller's workspace
  uint32_t *hist;            // [B][4096] scan: histogram of block maxima
  uint32_t *hist2;           // [B][4096] position scores' histogram
  uint32_t *smax;            // [B]   scan's max key scale (float bits)
  uint32_t *smax2;           // [B]   position stage's max key scale
  uint32_t *cand_cnt;        // [B]
  uint32_t *pcb_cnt;         // [B]
  float *bmax;               // [B][nbm]
  uint64_t *cand;            // [B][nbm]
  int32_t *pcb;              // [B][n_keep]
  float *pvals;              // [B][pv_stride] position scores (Reindex)
  float *sigma;              // [B][sigma_stride] the scan's position scores (Full)
  int32_t *unc_id;           // [B][3][unc_x] item lists that overflow shared memory
  float2 *unc_val;           // [B][unc_x] their exact scores as normalised double-floats
  int64_t nbm, unc_x;        // block maxima per sequence (a multiple of 4), overflow list length
  int64_t pv_stride;         // n_keep * block rounded up to a multiple of 4
  int64_t sigma_stride;      // nbm * block
  size_t zero_bytes;         // bytes at the start that must be zeroed per call
};

size_t indexer_ws_bytes(int32_t B, int64_t max_len, int32_t block, int32_t n_keep);
IndexerWs indexer_ws_carve(void *ws, int32_t B, int64_t max_len, int32_t block, int32_t n_keep);

cudaError_t launch_full_select(const csa2_cache &c, const uint16_t *q, const float *w, int block,
                               int n_keep, int topk, int64_t max_len, int32_t *pool, int32_t *topk_idx,
                               const IndexerWs &ws, int32_t *d_err, const csa2_profile *prof,
                               cudaStream_t st);
cudaError_t launch_reindex_select(const csa2_cache &c, const uint16_t *q, const float *w,
                                  const int32_t *pool, int block, int n_keep, int topk, int64_t max_len,
                                  int32_t *topk_idx, const IndexerWs &ws, int32_t *d_err, cudaStream_t st);
// Chunked-query scores on the tensor cores: rows [0, n) of a row view of the cache; groups
// of 16 rows sharing one base are scored, the others are left to the one-query scan.
struct CqArgs {
  const uint8_t *ik_codes;
  const float *ik_scale;
  const int64_t *base_v;     // [n] each row's session base
  const int32_t *len_v;      // [n] each row's length (position + 1; 0: none)
  const uint16_t *q;         // [n][8][64] bf16
  const float *w;            // [n][8]
  int n;
  IndexerWs ws;              // carved for >= n rows
  int32_t *d_err;
};
cudaError_t launch_chunk_scores_tc(const CqArgs &a, int block, cudaStream_t st);
cudaError_t launch_test_chunk_scores(const csa2_cache &c, const uint16_t *q, const float *w, const int32_t *q_seq,
                                     const int64_t *q_pos, int64_t T, int64_t max_len, float *sigma, double *bound,
                                     void *ws, int32_t *d_err, cudaStream_t st);
size_t chunked_ws_bytes(int64_t T, int64_t max_len, int32_t block, int32_t n_keep);
cudaError_t launch_chunked_select(const csa2_cache &c, const uint16_t *q, const float *w, const int32_t *q_seq,
                                  const int64_t *q_pos, int64_t T, int block, int n_keep, int topk, int64_t max_len,
                                  int32_t *pool, int32_t *topk_idx, void *ws, int32_t *d_err, cudaStream_t st);
cudaError_t launch_verify_select(const csa2_cache &c, const uint16_t *q, const float *w, const int32_t *q_seq,
                                 const int64_t *q_pos, int64_t T, const int32_t *pool, int block, int n_keep, int topk,
                                 int64_t max_len, int32_t *topk_idx, const IndexerWs &ws, int32_t *d_err,
                                 cudaStream_t st);
cudaError_t launch_test_scores(const csa2_cache &c, const uint16_t *q, const float *w, int64_t max_len,
                               float *sigma, double *bound, const IndexerWs &ws, int32_t *d_err,
                               cudaStream_t st);

// ---- attention ----
size_t attn_ws_bytes(int64_t T, int32_t H, int32_t topk, int32_t window);
cudaError_t launch_attn_decode(const csa2_cache &c, const csa2_swa &swa, const uint16_t *q, int H, int64_t T,
                               const int32_t *q_seq, const int64_t *q_pos, const int32_t *topk_idx,
                               int topk, int window, float tau, float *out, float *lse, void *ws,
                               int32_t *d_err, cudaStream_t st);

// chunked-query attention on tcgen05 (many rows, H <= 64)
bool attn_tc_eligible(int64_t T, int H);
cudaError_t launch_attn_chunked_tc(const csa2_cache &c, const csa2_swa &swa, const uint16_t *q, int H, int64_t T,
                                   const int32_t *q_seq, const int64_t *q_pos, const int32_t *topk_idx, int topk,
                                   int window, float tau, float *out, float *lse, int32_t *d_err, cudaStream_t st);

// ---- per-device launch facts (device_state.cu) ----
enum MemoSite {
  kSiteDeviceOk = 1,
  kSiteNumSms,
  kSiteScanOccupancy,
  kSiteScanOptin,
  kSiteSelectOptin,
  kSitePositionsResident,
  kSiteAttnOptin,
  kSiteAttnTcOptin,
  kSiteChunkScoresOptin,
};
// The value memoised for (device, site, key); make() computes it on first use (a negative
// result is not kept).  device_memo uses the current device.
int memo_lookup(int device, int site, int64_t key, const std::function<int()> &make);
int device_memo(int site, int64_t key, const std::function<int()> &make);
// Opt `kernel` in to `bytes` of dynamic shared memory on the current device, once.
int opt_in_smem(const void *kernel, size_t bytes, int site, int64_t key);
int num_sms();

}  // namespace csa2
