// Hierarchical sparse indexer: Full scan + block pool + top-k, Reindex over the pool.
//
// Method: origotech.dev deep dive, subsection "Compressed Sparse Attention 2(CSA2)":
// the first Full layer scores every cached position and keeps 2,048 blocks of 8
// positions plus its top-512; Reindex layers rescore only that pool with their own
// indexer queries; Reuse layers take the indices unchanged.
//
// Score of position t: sigma_t = s_t * sum_h w_h * max(q_h . k_t, 0), 8 heads of dim 64,
// k_t E4M3 values, s_t the key's float32 scale.
//
// Exact selection from approximate scores.  The scan computes q . k on the tensor
// cores (mma.sync m16n8k16: E4M3 keys converted exactly to f16, bf16 queries scaled by
// a power of two per head into f16, f32 accumulation).  Every approximate score obeys
//     |sigma~ - sigma| <= E + r * sigma~
// with E = s_max * 448 * sum_h w_h 2^-c_h (2^-16 ||q'_h||_1 + 64 * 2^-25) (the
// accumulation error of at most 2^-16 * sum|terms| over four chained k16 steps, plus the
// f16 conversion of the queries) and r = 2^-19 (epilogue rounding).  For a top-k by
// value, with theta~ the k-th largest approximate value, an item is certainly in if
// sigma~ > ((1+r) theta~ + 2E)/(1-r), certainly out if sigma~ < ((1-r) theta~ - 2E)/(1+r),
// and otherwise rescored in float64 (exact products, float64 sums) before the final
// choice by (score desc, id asc).
#include <cfloat>
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "launch.h"

namespace csa2 {

constexpr double kEpsAcc = 1.52587890625e-05;        // 2^-16
constexpr double kConvAbs = 64.0 * 2.98023223876953125e-08;  // 64 * 2^-25
constexpr double kRel = 1.9073486328125e-06;          // 2^-19
constexpr int kSelThreads = 1024;
constexpr int kMaxSel = 4096;                          // n_keep_blocks limit
constexpr int kMaxTopk = 1024;

// ------------------------------------------------------------------ query fragments

struct QFrag {
  uint32_t b[4][2];   // B operand: head g, dims 16t+4j .. 16t+4j+3 (f16, scaled by 2^c_g)
  float wi0, wi1;     // w_h * 2^-c_h for heads 2t, 2t+1
};

__device__ __forceinline__ int head_shift(float mx) {
  if (!(mx > 0.f)) return 0;
  int e = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;
  int c = 14 - e;
  return c < -60 ? -60 : (c > 60 ? 60 : c);
}

__device__ __forceinline__ float pow2f(int c) { return __uint_as_float((uint32_t)(c + 127) << 23); }

// 16 query values of head g at dims 16t..16t+15, as float, plus the head's shift
__device__ __forceinline__ int load_q16(const uint16_t *q_seq, int lane, float v[16]) {
  const int g = lane >> 2, t = lane & 3;
  const uint4 *p = reinterpret_cast<const uint4 *>(q_seq + g * kDIdx + 16 * t);
  uint4 r0 = __ldg(p), r1 = __ldg(p + 1);
  uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_to_f32(w[i] & 0xFFFFu);
    v[2 * i + 1] = bf16_to_f32(w[i] >> 16);
    mx = fmaxf(mx, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
  }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  return head_shift(mx);
}

__device__ __forceinline__ void load_qfrag(const uint16_t *q_seq, const float *w_seq, int lane, QFrag &f) {
  float v[16];
  const int c = load_q16(q_seq, lane, v);
  const float sc = pow2f(c);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f.b[j][0] = pack_f16x2(v[4 * j] * sc, v[4 * j + 1] * sc);
    f.b[j][1] = pack_f16x2(v[4 * j + 2] * sc, v[4 * j + 3] * sc);
  }
  const int t = lane & 3;
  const int c0 = __shfl_sync(0xffffffffu, c, 8 * t);
  const int c1 = __shfl_sync(0xffffffffu, c, 8 * t + 4);
  f.wi0 = __ldg(w_seq + 2 * t) * pow2f(-c0);
  f.wi1 = __ldg(w_seq + 2 * t + 1) * pow2f(-c1);
}

// Absolute error bound E of one sequence (identical in every lane).
__device__ double seq_bound(const uint16_t *q_seq, const float *w_seq, float smax, int lane) {
  float v[16];
  const int c = load_q16(q_seq, lane, v);
  const float sc = pow2f(c);
  double l1 = 0.0;
#pragma unroll
  for (int i = 0; i < 16; ++i) l1 += fabs((double)__half2float(__float2half_rn(v[i] * sc)));
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const int g = lane >> 2;
  double term = 0.0;
  if ((lane & 3) == 0)
    term = (double)__ldg(w_seq + g) * (double)pow2f(-c) * (kEpsAcc * 448.0 * l1 + kConvAbs * 448.0);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
  const double E = (double)smax * term * (1.0 + 1e-9) + (double)smax * 1e-30;
  return E > 0.0 ? E : 0.0;   // also maps NaN to 0
}

__device__ __forceinline__ float hi_cut(float theta, double E) {
  return __double2float_ru((1.0 + 4.0 * kRel) * (double)theta + 2.0 * E * (1.0 + 4.0 * kRel));
}
__device__ __forceinline__ float lo_cut(float theta, double E) {
  return __double2float_rd((1.0 - 4.0 * kRel) * (double)theta - 2.0 * E * (1.0 + 4.0 * kRel));
}

// ------------------------------------------------------------------ approximate scores

// Scores of 16 positions: row g and row g+8 of a 16-row tile; kg/kg8 hold key bytes
// 16t..16t+15 of those rows.  Each output is identical across the 4 lanes of a quad.
__device__ __forceinline__ void score16(const QFrag &f, const uint4 &kg, const uint4 &kg8, float sg,
                                        float sg8, float &og, float &og8) {
  float c[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t wg[4] = {kg.x, kg.y, kg.z, kg.w};
  const uint32_t w8[4] = {kg8.x, kg8.y, kg8.z, kg8.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t a0 = e4m3x2_to_f16x2(wg[j]), a2 = e4m3x2_to_f16x2(wg[j] >> 16);
    const uint32_t a1 = e4m3x2_to_f16x2(w8[j]), a3 = e4m3x2_to_f16x2(w8[j] >> 16);
    mma_16816(c, a0, a1, a2, a3, f.b[j][0], f.b[j][1]);
  }
  float pg = fmaxf(c[0], 0.f) * f.wi0 + fmaxf(c[1], 0.f) * f.wi1;
  float p8 = fmaxf(c[2], 0.f) * f.wi0 + fmaxf(c[3], 0.f) * f.wi1;
  pg += __shfl_xor_sync(0xffffffffu, pg, 1);
  p8 += __shfl_xor_sync(0xffffffffu, p8, 1);
  pg += __shfl_xor_sync(0xffffffffu, pg, 2);
  p8 += __shfl_xor_sync(0xffffffffu, p8, 2);
  og = pg * sg;
  og8 = p8 * sg8;
  og = og > 0.f ? og : 0.f;    // also maps NaN and -0 to +0
  og8 = og8 > 0.f ? og8 : 0.f;
}

// ------------------------------------------------------------------ exact rescoring

// float64 score of one position, computed by a whole warp (all lanes return it).
__device__ double exact_sigma(const uint16_t *q_seq, const float *w_seq, const uint8_t *key_row,
                              float scale, int lane) {
  const int h = lane >> 2, c = lane & 3;
  const uint4 *qp = reinterpret_cast<const uint4 *>(q_seq + h * kDIdx + 16 * c);
  uint4 q0 = __ldg(qp), q1 = __ldg(qp + 1);
  uint4 k = __ldg(reinterpret_cast<const uint4 *>(key_row + 16 * c));
  const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  const uint32_t kw[4] = {k.x, k.y, k.z, k.w};
  double acc = 0.0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const double qv = (double)bf16_to_f32((qw[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
    const double kv = (double)e4m3_to_f32((kw[i >> 2] >> (8 * (i & 3))) & 0xFFu);
    acc += qv * kv;
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  double t = (double)__ldg(w_seq + h) * (acc > 0.0 ? acc : 0.0);
  t += __shfl_xor_sync(0xffffffffu, t, 4);
  t += __shfl_xor_sync(0xffffffffu, t, 8);
  t += __shfl_xor_sync(0xffffffffu, t, 16);
  return (double)scale * t;
}

// ------------------------------------------------------------------ shared CTA helpers

struct SeqTable {             // per-call view of the sequences, validated
  int32_t len;
  int64_t base;
};

__device__ __forceinline__ SeqTable seq_entry(const csa2_cache &c, int b, int64_t max_len, int32_t *d_err) {
  SeqTable e;
  e.len = c.seq_len[b];
  e.base = c.seq_base[b];
  if (e.len < 0 || e.len > max_len || e.base < 0 || e.base + e.len > c.T_cap) {
    if (d_err) set_err(d_err, CSA2_DEVERR_LEN);
    e.len = 0;
  }
  return e;
}

// Block-wide k-th largest key (keys: uint32, larger is better; requires 1 <= k <= #keys).
template <class KeyFn>
__device__ uint32_t cta_kth_largest(int n, int k, KeyFn key, uint32_t *s_hist, int *s_misc) {
  uint32_t prefix = 0, mask = 0;
  int rem = k;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) s_hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
      const uint32_t kk = key(i);
      if ((kk & mask) == prefix) atomicAdd(&s_hist[(kk >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      int loc[8];
      int sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { loc[i] = (int)s_hist[255 - 8 * lane - i]; sum += loc[i]; }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int excl = incl - sum;
      if (excl < rem && rem <= incl) {
        for (int i = 0; i < 8; ++i) {
          if (excl + loc[i] >= rem) { s_misc[0] = 255 - 8 * lane - i; s_misc[1] = excl; break; }
          excl += loc[i];
        }
      }
    }
    __syncthreads();
    const uint32_t d = (uint32_t)s_misc[0];
    rem -= s_misc[1];
    prefix |= d << shift;
    mask |= 0xFFu << shift;
    __syncthreads();
  }
  return prefix;
}

// Ascending bitonic sort of s[0..n) in shared memory (n <= cap, cap a power of two).
__device__ void cta_sort_asc(int32_t *s, int n, int cap) {
  int N = 1;
  while (N < n) N <<= 1;
  for (int i = n + threadIdx.x; i < N; i += blockDim.x) s[i] = INT_MAX;
  __syncthreads();
  for (int size = 2; size <= N; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < N; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const int32_t a = s[i], b = s[j];
          if ((a > b) == up) { s[i] = b; s[j] = a; }
        }
      }
      __syncthreads();
    }
  }
  (void)cap;
}

__device__ __forceinline__ uint32_t value_key(float v) {   // v >= 0 -> bits+1, invalid (< 0) -> 0
  return v >= 0.f ? __float_as_uint(v) + 1u : 0u;
}

// ------------------------------------------------------------------ kernel arguments

struct IdxArgs {
  csa2_cache c;
  const uint16_t *q;        // [B][8][64]
  const float *w;           // [B][8]
  int64_t max_len;
  int32_t n_keep, topk;
  IndexerWs ws;
  int32_t *pool_out;        // [B][n_keep]
  const int32_t *pool_in;   // Reindex: [B][n_keep]
  int32_t *topk_out;        // [B][topk]
  float *sigma_out;         // test: [B][max_len]
  int32_t *d_err;
  int32_t use_pool;         // position stage reads pool_in instead of the candidate list
};

// ------------------------------------------------------------------ scan

constexpr int kScanWarps = 8;
constexpr int kScanDepth = 4;

template <int BLOCK>
__global__ void __launch_bounds__(kScanWarps * 32, 2) scan_kernel(const __grid_constant__ IdxArgs a) {
  __shared__ int64_t s_units[CSA2_MAX_B + 1];
  __shared__ int64_t s_base[CSA2_MAX_B];
  __shared__ int32_t s_len[CSA2_MAX_B];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = a.c.B;
  for (int i = tid; i < B; i += blockDim.x) {
    SeqTable e = seq_entry(a.c, i, a.max_len, blockIdx.x == 0 ? a.d_err : nullptr);
    s_len[i] = e.len;
    s_base[i] = e.base;
  }
  __syncthreads();
  if (warp == 0) {   // exclusive prefix of 16-position units per sequence
    const int per = (B + 31) / 32;
    int64_t local = 0;
    for (int i = lane * per; i < min(B, lane * per + per); ++i) local += (s_len[i] + 15) / 16;
    int64_t incl = local;
    for (int o = 1; o < 32; o <<= 1) {
      int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int64_t run = incl - local;
    for (int i = lane * per; i < min(B, lane * per + per); ++i) { s_units[i] = run; run += (s_len[i] + 15) / 16; }
    if (lane == 31) s_units[B] = incl;
  }
  __syncthreads();
  const int64_t total = s_units[B];
  const int64_t W = (int64_t)gridDim.x * kScanWarps;
  const int64_t gw = (int64_t)blockIdx.x * kScanWarps + warp;
  const int64_t per = (total + W - 1) / W;           // contiguous units per warp
  const int64_t u_begin = min(total, gw * per), u_end = min(total, u_begin + per);
  const int g = lane >> 2, t = lane & 3;

  struct Buf { uint4 kg, kg8; float sg, sg8; int b; int64_t p0; };
  Buf buf[kScanDepth];
  auto issue = [&](Buf &x, int64_t u) {
    x.b = -1;
    if (u >= u_end) return;
    int lo = 0, hi = B;             // s_units[lo] <= u < s_units[hi]
    while (hi - lo > 1) { int mid = (lo + hi) >> 1; if (s_units[mid] <= u) lo = mid; else hi = mid; }
    x.b = lo;
    x.p0 = (u - s_units[lo]) * 16;
    const int64_t L = s_len[lo], base = s_base[lo];
    const int64_t pg = x.p0 + g, pg8 = pg + 8;
    x.kg = make_uint4(0, 0, 0, 0);
    x.kg8 = make_uint4(0, 0, 0, 0);
    x.sg = 0.f;
    x.sg8 = 0.f;
    if (pg < L) { x.kg = ld_stream16(a.c.ik_codes + (base + pg) * kDIdx + 16 * t); x.sg = __ldg(a.c.ik_scale + base + pg); }
    if (pg8 < L) { x.kg8 = ld_stream16(a.c.ik_codes + (base + pg8) * kDIdx + 16 * t); x.sg8 = __ldg(a.c.ik_scale + base + pg8); }
  };

  QFrag f;
  int cur_b = -1;
  float smx = 0.f;
  auto flush = [&]() {
    if (cur_b >= 0) {
      float m = warp_max(smx);
      if (lane == 0) atomicMax(&a.ws.smax[cur_b], __float_as_uint(m));
    }
  };

#pragma unroll
  for (int d = 0; d < kScanDepth; ++d) issue(buf[d], u_begin + d);

  for (int64_t it = u_begin;; it += kScanDepth) {
    bool done = false;
#pragma unroll
    for (int d = 0; d < kScanDepth; ++d) {
      const int64_t u = it + d;
      if (u >= u_end) { done = true; break; }
      Buf x = buf[d];
      issue(buf[d], u + kScanDepth);
      const int b = x.b;
      if (b != cur_b) {
        flush();
        load_qfrag(a.q + (int64_t)b * kHIdx * kDIdx, a.w + (int64_t)b * kHIdx, lane, f);
        cur_b = b;
        smx = 0.f;
      }
      const int64_t L = s_len[b];
      float og, og8;
      score16(f, x.kg, x.kg8, x.sg, x.sg8, og, og8);
      smx = fmaxf(smx, fmaxf(x.sg, x.sg8));
      const int64_t pg = x.p0 + g, pg8 = pg + 8;
      if (a.sigma_out && t == 0) {
        if (pg < L) a.sigma_out[(int64_t)b * a.max_len + pg] = og;
        if (pg8 < L) a.sigma_out[(int64_t)b * a.max_len + pg8] = og8;
      }
      float *bmax = a.ws.bmax + (int64_t)b * a.ws.nbm;
      uint32_t *hist = a.ws.hist + (int64_t)b * kHistBins;
      if (BLOCK == 16) {
        float m = fmaxf(og, og8);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (lane == 0 && x.p0 < L) {
          bmax[x.p0 / 16] = m;
          atomicAdd(&hist[min(__float_as_uint(m) >> kHistShift, (uint32_t)kHistBins - 1)], 1u);
        }
      } else {
        float m = og, m8 = og8;
#pragma unroll
        for (int o = 4; o < 4 * BLOCK; o <<= 1) {
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          m8 = fmaxf(m8, __shfl_xor_sync(0xffffffffu, m8, o));
        }
        if (t == 0 && (g % BLOCK) == 0) {
          if (pg < L) {
            bmax[pg / BLOCK] = m;
            atomicAdd(&hist[min(__float_as_uint(m) >> kHistShift, (uint32_t)kHistBins - 1)], 1u);
          }
          if (pg8 < L) {
            bmax[pg8 / BLOCK] = m8;
            atomicAdd(&hist[min(__float_as_uint(m8) >> kHistShift, (uint32_t)kHistBins - 1)], 1u);
          }
        }
      }
    }
    if (done) break;
  }
  flush();
}

// ------------------------------------------------------------------ candidate collection

constexpr int kCollectPer = 4096;   // block maxima per CTA

__device__ float hist_threshold_low(const uint32_t *hist_g, int k, uint32_t *s_hist, int *s_misc) {
  // lower edge of the histogram bin holding the k-th largest block maximum
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) s_hist[i] = hist_g[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    const int per = kHistBins / 32;   // lane l owns bins [4096-per(l+1), 4096-per l), scanned top-down
    int sum = 0;
    for (int i = 0; i < per; ++i) sum += (int)s_hist[kHistBins - 1 - per * lane - i];
    int incl = sum;
    for (int o = 1; o < 32; o <<= 1) { int v = __shfl_up_sync(0xffffffffu, incl, o); if (lane >= o) incl += v; }
    int excl = incl - sum;
    if (excl < k && k <= incl) {
      for (int i = 0; i < per; ++i) {
        const int bin = kHistBins - 1 - per * lane - i;
        excl += (int)s_hist[bin];
        if (excl >= k) { s_misc[0] = bin; break; }
      }
    }
  }
  __syncthreads();
  const float th = __uint_as_float((uint32_t)s_misc[0] << kHistShift);
  __syncthreads();
  return th;
}

template <int BLOCK>
__global__ void __launch_bounds__(256) collect_kernel(const __grid_constant__ IdxArgs a) {
  __shared__ uint32_t s_hist[kHistBins];
  __shared__ int s_misc[4];
  __shared__ double s_E;
  const int b = blockIdx.y;
  const SeqTable e = seq_entry(a.c, b, a.max_len, nullptr);
  const int64_t nb = (e.len + BLOCK - 1) / BLOCK;
  const int64_t j0 = (int64_t)blockIdx.x * kCollectPer;
  if (j0 >= nb) return;
  float thr = -FLT_MAX;
  if (nb > a.n_keep) {
    if (threadIdx.x < 32) {
      double E = seq_bound(a.q + (int64_t)b * kHIdx * kDIdx, a.w + (int64_t)b * kHIdx,
                           __uint_as_float(a.ws.smax[b]), threadIdx.x);
      if (threadIdx.x == 0) s_E = E;
    }
    const float th_low = hist_threshold_low(a.ws.hist + (int64_t)b * kHistBins, a.n_keep, s_hist, s_misc);
    thr = lo_cut(th_low, s_E);
  }
  const float *bm = a.ws.bmax + (int64_t)b * a.ws.nbm;
  uint64_t *cand = a.ws.cand + (int64_t)b * a.ws.nbm;
  const int64_t j1 = min(nb, j0 + kCollectPer);
  const int64_t iters = (j1 - j0 + blockDim.x - 1) / blockDim.x;   // same trip count in every lane
  const int lane = threadIdx.x & 31;
  for (int64_t it = 0; it < iters; ++it) {
    const int64_t j = j0 + it * blockDim.x + threadIdx.x;
    const bool in = j < j1 && bm[j] >= thr;
    const unsigned mask = __ballot_sync(0xffffffffu, in);
    if (mask) {
      uint32_t base = 0;
      if (lane == 0) base = atomicAdd(&a.ws.cand_cnt[b], (uint32_t)__popc(mask));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (in) {
        const uint32_t off = base + __popc(mask & ((1u << lane) - 1u));
        cand[off] = ((uint64_t)__float_as_uint(bm[j]) << 32) | (uint32_t)j;
      }
    }
  }
}

// ------------------------------------------------------------------ block finalisation

template <int BLOCK>
__global__ void __launch_bounds__(kSelThreads) finalize_blocks_kernel(const __grid_constant__ IdxArgs a) {
  __shared__ uint32_t s_hist[256];
  __shared__ int s_misc[4];
  __shared__ int32_t s_sel[kMaxSel];
  __shared__ int s_cnt[4];
  __shared__ double s_E;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const SeqTable e = seq_entry(a.c, b, a.max_len, nullptr);
  const int64_t nb = (e.len + BLOCK - 1) / BLOCK;
  const int n_keep = a.n_keep;
  const int k1 = (int)min((int64_t)n_keep, nb);
  const int c = (int)a.ws.cand_cnt[b];
  const uint64_t *cand = a.ws.cand + (int64_t)b * a.ws.nbm;
  int32_t *pool = a.pool_out + (int64_t)b * n_keep;
  const uint16_t *qb = a.q + (int64_t)b * kHIdx * kDIdx;
  const float *wb = a.w + (int64_t)b * kHIdx;
  if (warp == 0) {
    double E = seq_bound(qb, wb, __uint_as_float(a.ws.smax[b]), lane);
    if (lane == 0) s_E = E;
  }
  if (tid < 4) s_cnt[tid] = 0;
  __syncthreads();
  const double E = s_E;
  auto cval = [&](int i) { return __uint_as_float((uint32_t)(cand[i] >> 32)); };
  auto cid = [&](int i) { return (int32_t)(uint32_t)cand[i]; };

  // ---- pool: top k1 blocks
  if (nb <= n_keep) {
    for (int i = tid; i < n_keep; i += blockDim.x) pool[i] = i < nb ? i : -1;
  } else {
    const uint32_t kth = cta_kth_largest(c, k1, [&](int i) { return value_key(cval(i)); }, s_hist, s_misc);
    const float theta = __uint_as_float(kth - 1u);
    const float hi = hi_cut(theta, E), lo = lo_cut(theta, E);
    int32_t *unc_id = a.ws.unc_id + (int64_t)b * a.ws.unc_cap;
    double *unc_val = a.ws.unc_val + (int64_t)b * a.ws.unc_cap;
    for (int i = tid; i < c; i += blockDim.x) {
      const float v = cval(i);
      if (v > hi) {
        const int slot = atomicAdd(&s_cnt[0], 1);
        if (slot < k1) s_sel[slot] = cid(i);
      } else if (v >= lo) {
        unc_id[atomicAdd(&s_cnt[1], 1)] = cid(i);
      }
    }
    __syncthreads();
    const int n_in = s_cnt[0], u = s_cnt[1];
    // exact block maxima of the uncertain blocks
    for (int i = warp; i < u; i += nwarps) {
      const int32_t j = unc_id[i];
      double best = -1.0;
      for (int r = 0; r < BLOCK; ++r) {
        const int64_t p = (int64_t)j * BLOCK + r;
        if (p >= e.len) break;
        const int64_t row = e.base + p;
        const double v = exact_sigma(qb, wb, a.c.ik_codes + row * kDIdx, __ldg(a.c.ik_scale + row), lane);
        best = fmax(best, v);
      }
      if (lane == 0) unc_val[i] = best;
    }
    __syncthreads();
    const int need = k1 - n_in;
    for (int i = tid; i < u; i += blockDim.x) {
      const double vi = unc_val[i];
      const int32_t ji = unc_id[i];
      int rank = 0;
      for (int m = 0; m < u; ++m) {
        const double vm = unc_val[m];
        rank += (vm > vi) || (vm == vi && unc_id[m] < ji);
      }
      if (rank < need) s_sel[n_in + rank] = ji;
    }
    __syncthreads();
    cta_sort_asc(s_sel, k1, kMaxSel);
    for (int i = tid; i < n_keep; i += blockDim.x) pool[i] = i < k1 ? s_sel[i] : -1;
  }
  __syncthreads();

  // ---- position-candidate blocks: every block that may hold a top-k position
  int32_t *pcb = a.ws.pcb + (int64_t)b * n_keep;
  if (nb <= a.topk) {
    for (int i = tid; i < nb; i += blockDim.x) pcb[i] = i;
    if (tid == 0) a.ws.pcb_cnt[b] = (uint32_t)nb;
  } else {
    const uint32_t kth = cta_kth_largest(c, a.topk, [&](int i) { return value_key(cval(i)); }, s_hist, s_misc);
    const float theta = __uint_as_float(kth - 1u);
    const float lo = lo_cut(theta, E);
    for (int i = tid; i < c; i += blockDim.x) {
      if (cval(i) >= lo) {
        const int slot = atomicAdd(&s_cnt[2], 1);
        if (slot < n_keep) pcb[slot] = cid(i);
      }
    }
    __syncthreads();
    if (s_cnt[2] > n_keep) {
      // a pathological band: fall back to the whole pool, which always contains them
      for (int i = tid; i < n_keep; i += blockDim.x) pcb[i] = pool[i];
      if (tid == 0) a.ws.pcb_cnt[b] = (uint32_t)n_keep;
    } else if (tid == 0) {
      a.ws.pcb_cnt[b] = (uint32_t)s_cnt[2];
    }
  }
}

// ------------------------------------------------------------------ position stage

// Approximate scores of the positions of a list of blocks (pcb or the pool).
template <int BLOCK>
__global__ void __launch_bounds__(256) score_positions_kernel(const __grid_constant__ IdxArgs a) {
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
  const SeqTable e = seq_entry(a.c, b, a.max_len, nullptr);
  const int64_t nb = (e.len + BLOCK - 1) / BLOCK;
  const int32_t *list;
  int count;
  if (a.use_pool) { list = a.pool_in + (int64_t)b * a.n_keep; count = a.n_keep; }
  else { list = a.ws.pcb + (int64_t)b * a.n_keep; count = (int)a.ws.pcb_cnt[b]; }
  const int n = count * BLOCK;
  const int units = (n + 15) / 16;
  float *pv = a.ws.pvals + (int64_t)b * a.n_keep * BLOCK;
  QFrag f;
  load_qfrag(a.q + (int64_t)b * kHIdx * kDIdx, a.w + (int64_t)b * kHIdx, lane, f);
  float smx = 0.f;
  for (int u = blockIdx.x * 8 + warp; u < units; u += gridDim.x * 8) {
    int64_t pos[2];
    uint4 k[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    float s[2] = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = u * 16 + g + 8 * h;
      pos[h] = -1;
      if (i < n) {
        const int32_t blk = list[i / BLOCK];
        if (blk >= 0) {
          if (blk >= nb) {
            if (t == 0) set_err(a.d_err, CSA2_DEVERR_POOL);
          } else {
            const int64_t p = (int64_t)blk * BLOCK + (i % BLOCK);
            if (p < e.len) pos[h] = p;
          }
        }
      }
      if (pos[h] >= 0) {
        const int64_t row = e.base + pos[h];
        k[h] = ld_nc16(a.c.ik_codes + row * kDIdx + 16 * t);
        s[h] = __ldg(a.c.ik_scale + row);
      }
    }
    float o0, o1;
    score16(f, k[0], k[1], s[0], s[1], o0, o1);
    smx = fmaxf(smx, fmaxf(s[0], s[1]));
    if (t == 0) {
      const int i0 = u * 16 + g;
      if (i0 < n) pv[i0] = pos[0] >= 0 ? o0 : -1.f;
      if (i0 + 8 < n) pv[i0 + 8] = pos[1] >= 0 ? o1 : -1.f;
    }
  }
  smx = warp_max(smx);
  if (lane == 0 && smx > 0.f) atomicMax(&a.ws.smax2[b], __float_as_uint(smx));
}

// Exact top-k positions from the approximate position scores.
template <int BLOCK>
__global__ void __launch_bounds__(kSelThreads) select_positions_kernel(const __grid_constant__ IdxArgs a) {
  __shared__ uint32_t s_hist[256];
  __shared__ int s_misc[4];
  __shared__ int32_t s_sel[kMaxTopk];
  __shared__ int s_cnt[4];
  __shared__ double s_E;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const SeqTable e = seq_entry(a.c, b, a.max_len, nullptr);
  const int32_t *list;
  int count;
  if (a.use_pool) { list = a.pool_in + (int64_t)b * a.n_keep; count = a.n_keep; }
  else { list = a.ws.pcb + (int64_t)b * a.n_keep; count = (int)a.ws.pcb_cnt[b]; }
  const int n = count * BLOCK;
  const float *pv = a.ws.pvals + (int64_t)b * a.n_keep * BLOCK;
  const uint16_t *qb = a.q + (int64_t)b * kHIdx * kDIdx;
  const float *wb = a.w + (int64_t)b * kHIdx;
  int32_t *out = a.topk_out + (int64_t)b * a.topk;
  auto pos_of = [&](int i) -> int64_t { return (int64_t)list[i / BLOCK] * BLOCK + (i % BLOCK); };
  if (tid < 4) s_cnt[tid] = 0;
  __syncthreads();
  int nv = 0;
  for (int i = tid; i < n; i += blockDim.x) nv += pv[i] >= 0.f;
  nv = __reduce_add_sync(0xffffffffu, nv);
  if (lane == 0) atomicAdd(&s_cnt[3], nv);
  __syncthreads();
  const int n_valid = s_cnt[3];
  const int k = min(a.topk, n_valid);
  if (n_valid <= a.topk) {
    for (int i = tid; i < n; i += blockDim.x)
      if (pv[i] >= 0.f) {
        const int slot = atomicAdd(&s_cnt[0], 1);
        if (slot < kMaxTopk) s_sel[slot] = (int32_t)pos_of(i);
      }
    __syncthreads();
  } else {
    if (warp == 0) {
      double E = seq_bound(qb, wb, __uint_as_float(a.ws.smax2[b]), lane);
      if (lane == 0) s_E = E;
    }
    const uint32_t kth = cta_kth_largest(n, k, [&](int i) { return value_key(pv[i]); }, s_hist, s_misc);
    const float theta = __uint_as_float(kth - 1u);
    const double E = s_E;
    const float hi = hi_cut(theta, E), lo = lo_cut(theta, E);
    int32_t *unc_id = a.ws.unc_id + (int64_t)b * a.ws.unc_cap;
    double *unc_val = a.ws.unc_val + (int64_t)b * a.ws.unc_cap;
    for (int i = tid; i < n; i += blockDim.x) {
      const float v = pv[i];
      if (v < 0.f) continue;
      if (v > hi) {
        const int slot = atomicAdd(&s_cnt[0], 1);
        if (slot < k) s_sel[slot] = (int32_t)pos_of(i);
      } else if (v >= lo) {
        unc_id[atomicAdd(&s_cnt[1], 1)] = (int32_t)pos_of(i);
      }
    }
    __syncthreads();
    const int n_in = s_cnt[0], u = s_cnt[1];
    for (int i = warp; i < u; i += nwarps) {
      const int64_t row = e.base + unc_id[i];
      const double v = exact_sigma(qb, wb, a.c.ik_codes + row * kDIdx, __ldg(a.c.ik_scale + row), lane);
      if (lane == 0) unc_val[i] = v;
    }
    __syncthreads();
    const int need = k - n_in;
    for (int i = tid; i < u; i += blockDim.x) {
      const double vi = unc_val[i];
      const int32_t pi = unc_id[i];
      int rank = 0;
      for (int m = 0; m < u; ++m) {
        const double vm = unc_val[m];
        rank += (vm > vi) || (vm == vi && unc_id[m] < pi);
      }
      if (rank < need) s_sel[n_in + rank] = pi;
    }
    __syncthreads();
  }
  cta_sort_asc(s_sel, k, kMaxTopk);
  for (int i = tid; i < a.topk; i += blockDim.x) out[i] = i < k ? s_sel[i] : -1;
}

// ------------------------------------------------------------------ test: bounds

__global__ void bound_kernel(const __grid_constant__ IdxArgs a, double *bound) {
  const int b = blockIdx.x;
  double E = seq_bound(a.q + (int64_t)b * kHIdx * kDIdx, a.w + (int64_t)b * kHIdx,
                       __uint_as_float(a.ws.smax[b]), threadIdx.x);
  if (threadIdx.x == 0) bound[b] = E;
  if (b == 0 && threadIdx.x == 0) bound[a.c.B] = kRel;
}

// ------------------------------------------------------------------ host side

static size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

size_t indexer_ws_bytes(int32_t B, int64_t max_len, int32_t block, int32_t n_keep) {
  const int64_t nbm = (max_len + block - 1) / block;
  const int64_t npos = (int64_t)n_keep * block;
  const int64_t unc = nbm > npos ? nbm : npos;
  size_t z = align_up((size_t)B * kHistBins * 4) + 4 * align_up((size_t)B * 4);
  size_t s = z;
  s += align_up((size_t)B * nbm * 4);       // bmax
  s += align_up((size_t)B * nbm * 8);       // cand
  s += align_up((size_t)B * n_keep * 4);    // pcb
  s += align_up((size_t)B * npos * 4);      // pvals
  s += align_up((size_t)B * unc * 4);       // unc_id
  s += align_up((size_t)B * unc * 8);       // unc_val
  return s;
}

IndexerWs indexer_ws_carve(void *ws, int32_t B, int64_t max_len, int32_t block, int32_t n_keep) {
  IndexerWs w;
  const int64_t nbm = (max_len + block - 1) / block;
  const int64_t npos = (int64_t)n_keep * block;
  w.nbm = nbm;
  w.unc_cap = nbm > npos ? nbm : npos;
  char *p = (char *)ws;
  w.hist = (uint32_t *)p; p += align_up((size_t)B * kHistBins * 4);
  w.smax = (uint32_t *)p; p += align_up((size_t)B * 4);
  w.smax2 = (uint32_t *)p; p += align_up((size_t)B * 4);
  w.cand_cnt = (uint32_t *)p; p += align_up((size_t)B * 4);
  w.pcb_cnt = (uint32_t *)p; p += align_up((size_t)B * 4);
  w.zero_bytes = (size_t)(p - (char *)ws);
  w.bmax = (float *)p; p += align_up((size_t)B * nbm * 4);
  w.cand = (uint64_t *)p; p += align_up((size_t)B * nbm * 8);
  w.pcb = (int32_t *)p; p += align_up((size_t)B * n_keep * 4);
  w.pvals = (float *)p; p += align_up((size_t)B * npos * 4);
  w.unc_id = (int32_t *)p; p += align_up((size_t)B * w.unc_cap * 4);
  w.unc_val = (double *)p;
  return w;
}

static int g_num_sms = 0;
int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  return g_num_sms;
}

// persistent scan grid: every resident CTA slot of the GPU, capped by the work
template <int BLOCK>
static int scan_grid_size(int B, int64_t max_len) {
  static int per_sm = 0;
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, scan_kernel<BLOCK>, kScanWarps * 32, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
  }
  const int64_t units_ub = (int64_t)B * ((max_len + 15) / 16);
  const int64_t g = std::min<int64_t>((units_ub + kScanWarps - 1) / kScanWarps, (int64_t)num_sms() * per_sm);
  return (int)std::max<int64_t>(g, 1);
}

template <int BLOCK>
static cudaError_t full_select_impl(IdxArgs &a, int64_t max_len, const csa2_profile *prof, cudaStream_t st) {
  const int B = a.c.B;
  const int scan_grid = scan_grid_size<BLOCK>(B, max_len);
  if (prof) cudaEventRecordWithFlags((cudaEvent_t)prof->start, st, cudaEventRecordExternal);
  scan_kernel<BLOCK><<<scan_grid, kScanWarps * 32, 0, st>>>(a);
  if (prof) cudaEventRecordWithFlags((cudaEvent_t)prof->stop, st, cudaEventRecordExternal);
  const int64_t nbm = a.ws.nbm;
  dim3 cg((unsigned)((nbm + kCollectPer - 1) / kCollectPer), (unsigned)B);
  collect_kernel<BLOCK><<<cg, 256, 0, st>>>(a);
  finalize_blocks_kernel<BLOCK><<<B, kSelThreads, 0, st>>>(a);
  const int per_seq = max(1, min(32, (int)((int64_t)num_sms() * 2 / max(B, 1))));
  score_positions_kernel<BLOCK><<<dim3(per_seq, B), 256, 0, st>>>(a);
  select_positions_kernel<BLOCK><<<B, kSelThreads, 0, st>>>(a);
  return cudaGetLastError();
}

template <int BLOCK>
static cudaError_t reindex_impl(IdxArgs &a, cudaStream_t st) {
  const int B = a.c.B;
  const int per_seq = max(1, min(32, (int)((int64_t)num_sms() * 2 / max(B, 1))));
  score_positions_kernel<BLOCK><<<dim3(per_seq, B), 256, 0, st>>>(a);
  select_positions_kernel<BLOCK><<<B, kSelThreads, 0, st>>>(a);
  return cudaGetLastError();
}

static IdxArgs make_args(const csa2_cache &c, const uint16_t *q, const float *w, int64_t max_len, int n_keep,
                         int topk, const IndexerWs &ws, int32_t *d_err) {
  IdxArgs a;
  a.c = c; a.q = q; a.w = w; a.max_len = max_len; a.n_keep = n_keep; a.topk = topk; a.ws = ws;
  a.pool_out = nullptr; a.pool_in = nullptr; a.topk_out = nullptr; a.sigma_out = nullptr;
  a.d_err = d_err; a.use_pool = 0;
  return a;
}

#define CSA2_DISPATCH_BLOCK(blk, call) \
  switch (blk) {                       \
    case 1: { constexpr int BL = 1; return call; } \
    case 2: { constexpr int BL = 2; return call; } \
    case 4: { constexpr int BL = 4; return call; } \
    case 8: { constexpr int BL = 8; return call; } \
    case 16: { constexpr int BL = 16; return call; } \
    default: return cudaErrorInvalidValue; \
  }

cudaError_t launch_full_select(const csa2_cache &c, const uint16_t *q, const float *w, int block, int n_keep,
                               int topk, int64_t max_len, int32_t *pool, int32_t *topk_idx, const IndexerWs &ws,
                               int32_t *d_err, const csa2_profile *prof, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(ws.hist, 0, ws.zero_bytes, st);
  if (e != cudaSuccess) return e;
  IdxArgs a = make_args(c, q, w, max_len, n_keep, topk, ws, d_err);
  a.pool_out = pool;
  a.pool_in = pool;
  a.topk_out = topk_idx;
  CSA2_DISPATCH_BLOCK(block, full_select_impl<BL>(a, max_len, prof, st));
}

cudaError_t launch_reindex_select(const csa2_cache &c, const uint16_t *q, const float *w, const int32_t *pool,
                                  int block, int n_keep, int topk, int64_t max_len, int32_t *topk_idx,
                                  const IndexerWs &ws, int32_t *d_err, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(ws.hist, 0, ws.zero_bytes, st);
  if (e != cudaSuccess) return e;
  IdxArgs a = make_args(c, q, w, max_len, n_keep, topk, ws, d_err);
  a.pool_in = pool;
  a.topk_out = topk_idx;
  a.use_pool = 1;
  CSA2_DISPATCH_BLOCK(block, reindex_impl<BL>(a, st));
}

cudaError_t launch_test_scores(const csa2_cache &c, const uint16_t *q, const float *w, int64_t max_len,
                               float *sigma, double *bound, const IndexerWs &ws, int32_t *d_err,
                               cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(ws.hist, 0, ws.zero_bytes, st);
  if (e != cudaSuccess) return e;
  IdxArgs a = make_args(c, q, w, max_len, 1, 1, ws, d_err);
  a.sigma_out = sigma;
  const int B = c.B;
  scan_kernel<8><<<scan_grid_size<8>(B, max_len), kScanWarps * 32, 0, st>>>(a);
  bound_kernel<<<B, 32, 0, st>>>(a, bound);
  return cudaGetLastError();
}

}  // namespace csa2
