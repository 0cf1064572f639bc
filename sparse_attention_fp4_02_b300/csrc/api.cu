// C ABI of the CSA2 library: host-side validation, workspace sizing, dispatch.
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "launch.h"

using namespace csa2;

namespace {

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

// compute capability 10.3 check, memoised per device
int device_ok() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  const int ok = device_memo(kSiteDeviceOk, 0, [dev] {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return -1;
    return (major == 10 && minor == 3) ? 1 : 0;
  });
  if (ok < 0) return CSA2_ERR_CUDA;
  return ok == 1 ? CSA2_OK : CSA2_ERR_UNSUPPORTED;
}

bool cache_ok(const csa2_cache *c) {
  if (!c) return false;
  if (!c->kv_codes || !c->kv_scales || !c->ik_codes || !c->ik_scale || !c->seq_base || !c->seq_len) return false;
  if (!aligned(c->kv_codes, 16) || !aligned(c->kv_scales, 16) || !aligned(c->ik_codes, 16) ||
      !aligned(c->ik_scale, 16) || !aligned(c->seq_base, 8) || !aligned(c->seq_len, 4))
    return false;
  return c->B >= 1 && c->B <= CSA2_MAX_B && c->T_cap >= 1 && c->T_cap <= (int64_t)INT32_MAX;
}

bool block_ok(int32_t block) { return block == 1 || block == 2 || block == 4 || block == 8 || block == 16; }

bool select_sizes_ok(int32_t B, int64_t max_len, int32_t block, int32_t n_keep, int32_t topk) {
  return B >= 1 && B <= CSA2_MAX_B && max_len >= 0 && max_len <= (int64_t)INT32_MAX && block_ok(block) &&
         n_keep >= 1 && n_keep <= 4096 && topk >= 1 && topk <= 1024 && topk <= n_keep;
}

bool attn_sizes_ok(int64_t T, int32_t H, int32_t topk, int32_t window) {
  return T >= 0 && T <= (int64_t)INT32_MAX && H >= 16 && H <= 128 && (H % 16) == 0 && topk >= 0 &&
         topk <= 4096 && window >= 0 && window <= 1024;
}

}  // namespace

extern "C" {

const char *csa2_status_string(int status) {
  switch (status) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case CSA2_ERR_UNSUPPORTED: return "unsupported device (needs compute capability 10.3)";
    case CSA2_ERR_CUDA: return "CUDA runtime or launch error";
    case CSA2_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int csa2_workspace_bytes(int op, int32_t B, int64_t max_len, int32_t block, int32_t n_keep_blocks, int32_t topk,
                         int64_t T, int32_t H, int32_t window, size_t *bytes) {
  if (!bytes) return CSA2_ERR_INVALID_ARG;
  switch (op) {
    case CSA2_OP_FULL_SELECT:
    case CSA2_OP_REINDEX_SELECT:
      if (!select_sizes_ok(B, max_len, block, n_keep_blocks, topk)) return CSA2_ERR_INVALID_ARG;
      *bytes = indexer_ws_bytes(B, max_len, block, n_keep_blocks);
      return CSA2_OK;
    case CSA2_OP_VERIFY_SELECT:
      if (T < 0 || T > 65535 || !select_sizes_ok(1, 0, block, n_keep_blocks, topk)) return CSA2_ERR_INVALID_ARG;
      *bytes = indexer_ws_bytes((int32_t)(T > 0 ? T : 1), 0, block, n_keep_blocks);
      return CSA2_OK;
    case CSA2_OP_CHUNKED_SELECT:
      if (T < 0 || T > (1 << 24) || !select_sizes_ok(1, max_len, block, n_keep_blocks, topk))
        return CSA2_ERR_INVALID_ARG;
      *bytes = chunked_ws_bytes(T, max_len, block, n_keep_blocks);
      return CSA2_OK;
    case CSA2_OP_ATTN_DECODE:
      if (!attn_sizes_ok(T, H, topk, window)) return CSA2_ERR_INVALID_ARG;
      *bytes = attn_ws_bytes(T, H, topk, window);
      return CSA2_OK;
    default:
      return CSA2_ERR_INVALID_ARG;
  }
}

int kv_append_fp4(const csa2_cache *cache, const csa2_swa *swa_layers, int32_t n_swa_layers,
                  const uint16_t *kv_new, const uint16_t *ik_new, const uint16_t *swa_new, const float *rope_cos,
                  const float *rope_sin, int64_t rope_len, const int32_t *seq_id, const int64_t *pos, int64_t n,
                  int32_t *d_err, csa2_stream_t stream) {
  if (!cache_ok(cache) || n < 0 || !d_err) return CSA2_ERR_INVALID_ARG;
  if (n_swa_layers < 0 || n_swa_layers > CSA2_MAX_SWA_LAYERS) return CSA2_ERR_INVALID_ARG;
  if (n > 0) {
    if (!kv_new || !aligned(kv_new, 8) || !rope_cos || !rope_sin || rope_len < 1 || !seq_id || !pos)
      return CSA2_ERR_INVALID_ARG;
    if (ik_new && !aligned(ik_new, 4)) return CSA2_ERR_INVALID_ARG;
    if (swa_new) {
      if (!aligned(swa_new, 8) || n_swa_layers < 1 || !swa_layers) return CSA2_ERR_INVALID_ARG;
      for (int l = 0; l < n_swa_layers; ++l) {
        const csa2_swa &w = swa_layers[l];
        if (!w.codes || !w.scale || w.ring < 1 || !aligned(w.codes, 16) || !aligned(w.scale, 4))
          return CSA2_ERR_INVALID_ARG;
      }
    }
  }
  int st = device_ok();
  if (st != CSA2_OK) return st;
  return cuda_status(launch_append(*cache, swa_layers, swa_new ? n_swa_layers : 0, kv_new, ik_new, swa_new,
                                   rope_cos, rope_sin, rope_len, seq_id, pos, n, d_err, (cudaStream_t)stream));
}

int swa_refill_fp8(const csa2_swa *swa_layers, int32_t n_swa_layers, int32_t B, const uint16_t *swa_new,
                   const float *rope_cos, const float *rope_sin, int64_t rope_len, const int32_t *seq_id,
                   const int64_t *pos, int64_t n, int32_t *d_err, csa2_stream_t stream) {
  if (n < 0 || !d_err || B < 1 || B > CSA2_MAX_B) return CSA2_ERR_INVALID_ARG;
  if (n_swa_layers < 1 || n_swa_layers > CSA2_MAX_SWA_LAYERS || !swa_layers) return CSA2_ERR_INVALID_ARG;
  for (int l = 0; l < n_swa_layers; ++l) {
    const csa2_swa &w = swa_layers[l];
    if (!w.codes || !w.scale || w.ring < 1 || !aligned(w.codes, 16) || !aligned(w.scale, 4))
      return CSA2_ERR_INVALID_ARG;
  }
  if (n > 0 && (!swa_new || !aligned(swa_new, 8) || !rope_cos || !rope_sin || rope_len < 1 || !seq_id || !pos))
    return CSA2_ERR_INVALID_ARG;
  int st = device_ok();
  if (st != CSA2_OK) return st;
  csa2_cache none;
  std::memset(&none, 0, sizeof(none));
  none.B = B;                                                // sequence ids are checked against B only
  return cuda_status(launch_append(none, swa_layers, n_swa_layers, nullptr, nullptr, swa_new, rope_cos, rope_sin,
                                   rope_len, seq_id, pos, n, d_err, (cudaStream_t)stream));
}

int indexer_full_select(const csa2_cache *cache, const uint16_t *q_idx, const float *w, int32_t block,
                        int32_t n_keep_blocks, int32_t topk, int64_t max_len, int32_t *pool_blocks,
                        int32_t *topk_idx, void *ws, size_t ws_bytes, int32_t *d_err, const csa2_profile *prof,
                        csa2_stream_t stream) {
  if (!cache_ok(cache) || !q_idx || !aligned(q_idx, 16) || !w || !aligned(w, 4) || !pool_blocks ||
      !topk_idx || !d_err)
    return CSA2_ERR_INVALID_ARG;
  if (!select_sizes_ok(cache->B, max_len, block, n_keep_blocks, topk)) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < indexer_ws_bytes(cache->B, max_len, block, n_keep_blocks))
    return CSA2_ERR_WORKSPACE;
  int st = device_ok();
  if (st != CSA2_OK) return st;
  IndexerWs iw = indexer_ws_carve(ws, cache->B, max_len, block, n_keep_blocks);
  return cuda_status(launch_full_select(*cache, q_idx, w, block, n_keep_blocks, topk, max_len, pool_blocks,
                                        topk_idx, iw, d_err, prof, (cudaStream_t)stream));
}

int indexer_reindex_select(const csa2_cache *cache, const uint16_t *q_idx, const float *w,
                           const int32_t *pool_blocks, int32_t block, int32_t n_keep_blocks, int32_t topk,
                           int64_t max_len, int32_t *topk_idx, void *ws, size_t ws_bytes, int32_t *d_err,
                           csa2_stream_t stream) {
  if (!cache_ok(cache) || !q_idx || !aligned(q_idx, 16) || !w || !aligned(w, 4) || !pool_blocks || !topk_idx ||
      !d_err)
    return CSA2_ERR_INVALID_ARG;
  if (!select_sizes_ok(cache->B, max_len, block, n_keep_blocks, topk)) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < indexer_ws_bytes(cache->B, max_len, block, n_keep_blocks))
    return CSA2_ERR_WORKSPACE;
  int st = device_ok();
  if (st != CSA2_OK) return st;
  IndexerWs iw = indexer_ws_carve(ws, cache->B, max_len, block, n_keep_blocks);
  return cuda_status(launch_reindex_select(*cache, q_idx, w, pool_blocks, block, n_keep_blocks, topk, max_len,
                                           topk_idx, iw, d_err, (cudaStream_t)stream));
}

int indexer_chunked_select(const csa2_cache *cache, const uint16_t *q_idx, const float *w, const int32_t *q_seq,
                           const int64_t *q_pos, int64_t T, int32_t block, int32_t n_keep_blocks, int32_t topk,
                           int64_t max_len, int32_t *pool_blocks, int32_t *topk_idx, void *ws, size_t ws_bytes,
                           int32_t *d_err, csa2_stream_t stream) {
  if (!cache_ok(cache) || !d_err || T < 0 || T > (1 << 24)) return CSA2_ERR_INVALID_ARG;
  if (!select_sizes_ok(1, max_len, block, n_keep_blocks, topk)) return CSA2_ERR_INVALID_ARG;
  if (T == 0) return CSA2_OK;
  if (!q_idx || !aligned(q_idx, 16) || !w || !aligned(w, 4) || !q_seq || !q_pos || !pool_blocks || !topk_idx)
    return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < chunked_ws_bytes(T, max_len, block, n_keep_blocks))
    return CSA2_ERR_WORKSPACE;
  int st = device_ok();
  if (st != CSA2_OK) return st;
  return cuda_status(launch_chunked_select(*cache, q_idx, w, q_seq, q_pos, T, block, n_keep_blocks, topk, max_len,
                                           pool_blocks, topk_idx, ws, d_err, (cudaStream_t)stream));
}

int indexer_verify_select(const csa2_cache *cache, const uint16_t *q_idx, const float *w, const int32_t *q_seq,
                          const int64_t *q_pos, int64_t T, const int32_t *pool_blocks, int32_t block,
                          int32_t n_keep_blocks, int32_t topk, int64_t max_len, int32_t *topk_idx, void *ws,
                          size_t ws_bytes, int32_t *d_err, csa2_stream_t stream) {
  if (!cache_ok(cache) || !d_err || T < 0 || T > 65535) return CSA2_ERR_INVALID_ARG;
  if (!select_sizes_ok(cache->B, max_len, block, n_keep_blocks, topk)) return CSA2_ERR_INVALID_ARG;
  if (T == 0) return CSA2_OK;
  if (!q_idx || !aligned(q_idx, 16) || !w || !aligned(w, 4) || !q_seq || !q_pos || !pool_blocks || !topk_idx)
    return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < indexer_ws_bytes((int32_t)T, 0, block, n_keep_blocks))
    return CSA2_ERR_WORKSPACE;
  int st = device_ok();
  if (st != CSA2_OK) return st;
  IndexerWs iw = indexer_ws_carve(ws, (int32_t)T, 0, block, n_keep_blocks);
  return cuda_status(launch_verify_select(*cache, q_idx, w, q_seq, q_pos, T, pool_blocks, block, n_keep_blocks, topk,
                                          max_len, topk_idx, iw, d_err, (cudaStream_t)stream));
}

int sparse_attn_decode(const csa2_cache *cache, const csa2_swa *swa, const uint16_t *q, int32_t H, int64_t T,
                       const int32_t *q_seq, const int64_t *q_pos, const int32_t *topk_idx, int32_t topk,
                       int32_t window, float softmax_scale, float *out, float *lse, void *ws, size_t ws_bytes,
                       int32_t *d_err, csa2_stream_t stream) {
  if (!cache_ok(cache) || !swa || !d_err) return CSA2_ERR_INVALID_ARG;
  if (!attn_sizes_ok(T, H, topk, window)) return CSA2_ERR_INVALID_ARG;
  if (T > 0) {
    if (!q || !aligned(q, 16) || !q_seq || !q_pos || !out || !aligned(out, 16)) return CSA2_ERR_INVALID_ARG;
    if (topk > 0 && !topk_idx) return CSA2_ERR_INVALID_ARG;
    if (window > 0 && (!swa->codes || !swa->scale || swa->ring < window || !aligned(swa->codes, 16)))
      return CSA2_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f)) return CSA2_ERR_INVALID_ARG;
  }
  (void)ws;
  (void)ws_bytes;   // the kernel needs no workspace
  int st = device_ok();
  if (st != CSA2_OK) return st;
  csa2_swa sw = *swa;
  if (window == 0) { sw.ring = 1; }
  return cuda_status(launch_attn_decode(*cache, sw, q, H, T, q_seq, q_pos, topk_idx, topk, window, softmax_scale,
                                        out, lse, ws, d_err, (cudaStream_t)stream));
}

}  // extern "C"

// ---- workspace-free Reindex: scratch in a static device array ----------------------
namespace {

// Scratch of indexer_reindex_select_static.  In host code this name is only a handle
// for cudaGetSymbolAddress, never a device address.
__device__ __align__(256) unsigned char g_reindex_scratch[CSA2_STATIC_SCRATCH_BYTES];

// The array's device address on the current device, resolved once per device (with that
// device current) and kept beside the library's other per-device facts.
int static_scratch(void **out) {
  static std::mutex mu;
  static void *addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  if (dev < 0 || dev >= 64) return CSA2_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_reindex_scratch) != cudaSuccess || !p) return CSA2_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return CSA2_OK;
}

}  // namespace

extern "C" {

int indexer_reindex_select_static(const csa2_cache *cache, const uint16_t *q_idx, const float *w,
                                  const int32_t *pool_blocks, int32_t block, int32_t n_keep_blocks, int32_t topk,
                                  int64_t max_len, int32_t *topk_idx, int32_t *d_err, csa2_stream_t stream) {
  if (!cache_ok(cache) || !q_idx || !aligned(q_idx, 16) || !w || !aligned(w, 4) || !pool_blocks || !topk_idx ||
      !d_err)
    return CSA2_ERR_INVALID_ARG;
  if (!select_sizes_ok(cache->B, max_len, block, n_keep_blocks, topk)) return CSA2_ERR_INVALID_ARG;
  // a Reindex call touches no per-block arrays, so its layout is the one for max_len 0
  if (indexer_ws_bytes(cache->B, 0, block, n_keep_blocks) > (size_t)CSA2_STATIC_SCRATCH_BYTES)
    return CSA2_ERR_WORKSPACE;
  int st = device_ok();
  if (st != CSA2_OK) return st;
  void *scratch = nullptr;
  st = static_scratch(&scratch);
  if (st != CSA2_OK) return st;
  IndexerWs iw = indexer_ws_carve(scratch, cache->B, 0, block, n_keep_blocks);
  return cuda_status(launch_reindex_select(*cache, q_idx, w, pool_blocks, block, n_keep_blocks, topk, max_len,
                                           topk_idx, iw, d_err, (cudaStream_t)stream));
}

int csa2_test_quantize_fp4(const float *x, int64_t n_groups, uint8_t *codes, uint8_t *scales, csa2_stream_t stream) {
  if (n_groups < 0 || (n_groups > 0 && (!x || !aligned(x, 16) || !codes || !aligned(codes, 2) || !scales)))
    return CSA2_ERR_INVALID_ARG;
  int st = device_ok();
  if (st != CSA2_OK) return st;
  return cuda_status(launch_test_fp4(x, n_groups, codes, scales, (cudaStream_t)stream));
}

int csa2_test_quantize_fp8(const float *x, int64_t n, int32_t C, uint8_t *codes, float *scale, csa2_stream_t stream) {
  if (n < 0 || (C != 64 && C != 128) || (n > 0 && (!x || !codes || !scale))) return CSA2_ERR_INVALID_ARG;
  int st = device_ok();
  if (st != CSA2_OK) return st;
  return cuda_status(launch_test_fp8(x, n, C, codes, scale, (cudaStream_t)stream));
}

int csa2_test_index_scores(const csa2_cache *cache, const uint16_t *q_idx, const float *w, int64_t max_len,
                           float *sigma, double *bound, void *ws, size_t ws_bytes, int32_t *d_err,
                           csa2_stream_t stream) {
  if (!cache_ok(cache) || !q_idx || !aligned(q_idx, 16) || !w || !sigma || !bound || !d_err)
    return CSA2_ERR_INVALID_ARG;
  if (!select_sizes_ok(cache->B, max_len, 8, 1, 1)) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < indexer_ws_bytes(cache->B, max_len, 8, 1)) return CSA2_ERR_WORKSPACE;
  int st = device_ok();
  if (st != CSA2_OK) return st;
  IndexerWs iw = indexer_ws_carve(ws, cache->B, max_len, 8, 1);
  return cuda_status(launch_test_scores(*cache, q_idx, w, max_len, sigma, bound, iw, d_err, (cudaStream_t)stream));
}

int csa2_test_chunk_scores(const csa2_cache *cache, const uint16_t *q_idx, const float *w, const int32_t *q_seq,
                           const int64_t *q_pos, int64_t T, int64_t max_len, float *sigma, double *bound, void *ws,
                           size_t ws_bytes, int32_t *d_err, csa2_stream_t stream) {
  if (!cache_ok(cache) || !q_idx || !aligned(q_idx, 16) || !w || !q_seq || !q_pos || !sigma || !bound || !d_err ||
      T < 1 || T > CSA2_MAX_B)
    return CSA2_ERR_INVALID_ARG;
  if (!select_sizes_ok(1, max_len, 8, 1, 1)) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < chunked_ws_bytes(T, max_len, 8, 1)) return CSA2_ERR_WORKSPACE;
  int st = device_ok();
  if (st != CSA2_OK) return st;
  return cuda_status(launch_test_chunk_scores(*cache, q_idx, w, q_seq, q_pos, T, max_len, sigma, bound, ws, d_err,
                                              (cudaStream_t)stream));
}

}  // extern "C"
