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
// and otherwise rescored exactly before the final choice by (score desc, id asc): each
// head's dot product as a sum of exact integer products in 64-bit fixed point, then ReLU,
// head weights and the key scale in double-float (float pairs with error-free TwoSum and
// TwoProduct, 48 significant bits).
#include <cfloat>
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace csa2 {

constexpr float kEpsAcc448 = 448.0f * 0x1p-16f;      // 448 * 2^-16 (accumulation, relative to sum |terms|)
constexpr float kConvAbs448 = 448.0f * 64.0f * 0x1p-25f;   // 448 * 64 * 2^-25 (queries below the f16 range)
constexpr float kRelF = 0x1p-19f;                     // r = 2^-19
constexpr int kMaxSel = 4096;                          // n_keep_blocks limit

// ------------------------------------------------------------------ query fragments

struct QFrag {
  uint32_t b[4][2];   // B operand: head g, dims 16t+4j .. 16t+4j+3 (f16, scaled by 2^c_g)
  float wi0, wi1;     // w_h * 2^-c_h for heads 2t, 2t+1
};

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

// Absolute error bound E of one sequence (identical in every lane), rounded upward at
// every step so that the float result is never below the exact bound.
__device__ float seq_bound(const uint16_t *q_seq, const float *w_seq, float smax, int lane) {
  float v[16];
  const int c = load_q16(q_seq, lane, v);
  const float sc = pow2f(c);
  float l1 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) l1 = __fadd_ru(l1, fabsf(__half2float(__float2half_rn(v[i] * sc))));
  l1 = __fadd_ru(l1, __shfl_xor_sync(0xffffffffu, l1, 1));
  l1 = __fadd_ru(l1, __shfl_xor_sync(0xffffffffu, l1, 2));
  const int g = lane >> 2;
  float term = 0.f;
  if ((lane & 3) == 0)
    term = __fmul_ru(__fmul_ru(__ldg(w_seq + g), pow2f(-c)), __fadd_ru(__fmul_ru(kEpsAcc448, l1), kConvAbs448));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) term = __fadd_ru(term, __shfl_xor_sync(0xffffffffu, term, o));
  const float E = __fadd_ru(__fmul_ru(__fmul_ru(smax, term), 1.0f + 0x1p-20f), smax * 1e-30f);
  return E > 0.f ? E : 0.f;   // also maps NaN to 0
}

// Cuts of a threshold theta: every item above hi_cut is certainly above an item whose
// approximate value is theta, every item below lo_cut certainly below (the bound is
// |approx - exact| <= E + r * approx; the cuts take 4r for margin and round outward).
__device__ __forceinline__ float hi_cut(float theta, float E) {
  return __fadd_ru(__fmul_ru(1.0f + 4.0f * kRelF, theta), __fmul_ru(2.0f + 8.0f * kRelF, E));
}
__device__ __forceinline__ float lo_cut(float theta, float E) {
  return __fsub_rd(__fmul_rd(1.0f - 4.0f * kRelF, theta), __fmul_ru(2.0f + 8.0f * kRelF, E));
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

// Knuth's TwoSum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Double-float arithmetic (a value is hi + lo, |lo| <= ulp(hi)/2 after normalising).
__device__ __forceinline__ float2 df_norm(float a, float b) {
  float s, e;
  two_sum(a, b, s, e);
  return make_float2(s, e);
}
__device__ __forceinline__ float2 df_add(float2 a, float2 b) {
  float s, e;
  two_sum(a.x, b.x, s, e);
  return df_norm(s, __fadd_rn(e, __fadd_rn(a.y, b.y)));
}
__device__ __forceinline__ float2 df_mul(float2 a, float b) {     // TwoProduct through FMA
  const float p = __fmul_rn(a.x, b);
  const float e = __fmaf_rn(a.y, b, __fmaf_rn(a.x, b, -p));
  return df_norm(p, e);
}
__device__ __forceinline__ bool df_greater(float2 a, float2 b) { return a.x > b.x || (a.x == b.x && a.y > b.y); }
__device__ __forceinline__ bool df_equal(float2 a, float2 b) { return a.x == b.x && a.y == b.y; }

// Exact dot products in 64-bit integers.  k * 512 is an integer for every E4M3 value k
// (|k * 512| <= 229,376); each head's queries are rounded once to integers
// Q = RN(q * 2^(c_h + 15)), |Q| < 2^30, which is exact for every query value at least
// 2^-15 of the head scale 2^-c_h.  A head's 64 products then add exactly in int64; the
// sum, converted to a double-float, goes through the ReLU, head weights, head sum and key
// scale in double-float arithmetic (relative error about 2^-44).  No float64 instruction.
struct QExact {          // lane (h, c): head h's integer queries at dims 16c..16c+15
  int32_t Q[16];
  int sh;                // dot product = integer sum * 2^-sh
  float w;               // w_h
};

__device__ __forceinline__ void load_qexact(const uint16_t *q_seq, const float *w_seq, int lane, QExact &q) {
  float v[16];
  const int c_h = load_q16(q_seq, lane, v);
  const float sc = pow2f(c_h + 15);
#pragma unroll
  for (int i = 0; i < 16; ++i) q.Q[i] = __float2int_rn(v[i] * sc);
  q.sh = c_h + 24;
  q.w = __ldg(w_seq + (lane >> 2));
}

// E4M3 code -> code value * 512 (an integer); NaN codes map to 0
__device__ __forceinline__ void fill_e4m3_lut(int32_t *lut) {
  for (int c = threadIdx.x; c < 256; c += blockDim.x) {
    const float v = e4m3_to_f32((uint32_t)c) * 512.f;
    lut[c] = (v == v) ? __float2int_rn(v) : 0;
  }
}

// Score of one position, computed by a whole warp (all lanes return it) from the lane's
// 16 key bytes (dims 16c..16c+15) and the row's scale.
__device__ float2 exact_sigma(const QExact &q, const uint4 &k, float scale, const int32_t *lut) {
  const uint32_t kw[4] = {k.x, k.y, k.z, k.w};
  long long acc = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc += (long long)q.Q[4 * j + i] * (long long)lut[(kw[j] >> (8 * i)) & 0xFFu];
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  const float hi = __ll2float_rn(acc);
  const float lo = __ll2float_rn(acc - __float2ll_rz(hi));
  const float inv = pow2f(-q.sh);
  float2 d = df_norm(__fmul_rn(hi, inv), __fmul_rn(lo, inv));         // exact power-of-two scaling
  if (d.x < 0.f || (d.x == 0.f && d.y <= 0.f)) d = make_float2(0.f, 0.f);
  float2 t = df_mul(d, q.w);
#pragma unroll
  for (int o = 4; o <= 16; o <<= 1) {
    const float2 u = make_float2(__shfl_xor_sync(0xffffffffu, t.x, o), __shfl_xor_sync(0xffffffffu, t.y, o));
    t = df_add(t, u);
  }
  return df_mul(t, scale);
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

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += x;
  }
  return v;
}

// CTA-wide exclusive offset of each thread's `v` in thread order; s_scan needs 65 ints.
// Returns the exclusive offset; the total is left in s_scan[64].
__device__ __forceinline__ int cta_excl_scan(int v, int *s_scan) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int incl = warp_incl_scan(v);
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int x = lane < nw ? s_scan[lane] : 0;
    const int inc = warp_incl_scan(x);
    if (lane < nw) s_scan[32 + lane] = inc - x;
    if (lane == 31) s_scan[64] = inc;
  }
  __syncthreads();
  const int r = s_scan[32 + warp] + incl - v;
  __syncthreads();
  return r;
}

// Top-down search over `nbins` bin counts: the bin where the running count from the top
// first reaches k (1 <= k <= total).  s_out[0] = bin, s_out[1] = count strictly above it.
template <class CountFn>
__device__ void cta_find_bin(int nbins, int k, CountFn count, int *s_scan, int *s_out) {
  const int per = (nbins + blockDim.x - 1) / blockDim.x;
  const int top = nbins - 1 - (int)threadIdx.x * per;          // this thread's highest bin
  int sum = 0;
  for (int i = 0; i < per; ++i)
    if (top - i >= 0) sum += (int)count(top - i);
  int excl = cta_excl_scan(sum, s_scan);
  if (excl < k && k <= excl + sum) {
    for (int i = 0; i < per; ++i) {
      const int bin = top - i;
      const int cb = (int)count(bin);
      if (excl + cb >= k) { s_out[0] = bin; s_out[1] = excl; break; }
      excl += cb;
    }
  }
  __syncthreads();
}

// k-th largest key among the keys whose top 12 bits equal `bin` (1 <= k <= their number):
// two radix passes over the low 19 bits, lanes hitting the same bin add once (match_any).
template <class KeyFn>
__device__ uint32_t cta_kth_in_bin(int n, int k, KeyFn key, uint32_t bin, uint32_t *s_hist, int *s_scan,
                                   int *s_out) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int iters = (n + blockDim.x - 1) / blockDim.x;
  uint32_t prefix = bin;                                        // key >> 19
  int shift = kHistShift, width = 10;
  for (int pass = 0; pass < 2; ++pass) {
    const int nb = 1 << width;
    const int sub_shift = shift - width;
    for (int i = tid; i < nb; i += blockDim.x) s_hist[i] = 0u;
    __syncthreads();
    for (int it = 0; it < iters; ++it) {
      const int i = it * blockDim.x + tid;
      uint32_t kk = 0;
      bool in = false;
      if (i < n) { kk = key(i); in = (kk >> shift) == prefix; }
      const unsigned act = __ballot_sync(0xffffffffu, in);
      if (in) {
        const uint32_t sb = (kk >> sub_shift) & (uint32_t)(nb - 1);
        const unsigned grp = __match_any_sync(act, sb);
        if (lane == __ffs(grp) - 1) atomicAdd(&s_hist[sb], (uint32_t)__popc(grp));
      }
    }
    __syncthreads();
    cta_find_bin(nb, k, [&](int b) { return s_hist[b]; }, s_scan, s_out);
    prefix = (prefix << width) | (uint32_t)s_out[0];
    k -= s_out[1];
    shift = sub_shift;
    width = sub_shift;                                          // second pass: the last 9 bits
    __syncthreads();
  }
  return prefix;
}

// Warp-aggregated slot reservation on a shared counter (call with every lane of the warp).
__device__ __forceinline__ int warp_reserve(bool pred, int *counter) {
  const unsigned m = __ballot_sync(0xffffffffu, pred);
  const int lane = threadIdx.x & 31;
  int base = 0;
  if (m && lane == __ffs(m) - 1) base = atomicAdd(counter, __popc(m));
  base = __shfl_sync(0xffffffffu, base, __ffs(m ? m : 1u) - 1);
  return pred ? base + __popc(m & ((1u << lane) - 1u)) : -1;
}

// Ascending bitonic sort of s[0..n) in shared memory (n <= the buffer, a power of two).
__device__ void cta_sort_asc(int32_t *s, int n) {
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
}

// Writes map(i) for the set bits i of s_bits[0..nwords), ascending, to out[0..), then -1
// up to out[pad).  Returns the number of set bits.  Every thread of the CTA must call it.
template <class MapFn>
__device__ int emit_bits_ascending(const uint32_t *s_bits, int nwords, MapFn map, int32_t *out, int pad,
                                   int *s_scan) {
  const int tid = threadIdx.x;
  const int per = (nwords + blockDim.x - 1) / blockDim.x;
  const int w0 = min(nwords, tid * per), w1 = min(nwords, w0 + per);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(s_bits[w]);
  int pos = cta_excl_scan(cnt, s_scan);
  const int total = s_scan[64];
  for (int w = w0; w < w1; ++w) {
    uint32_t bits = s_bits[w];
    while (bits) {
      const int bit = __ffs(bits) - 1;
      bits &= bits - 1;
      if (pos < pad) out[pos] = map(w * 32 + bit);
      ++pos;
    }
  }
  for (int i = total + tid; i < pad; i += blockDim.x) out[i] = -1;
  __syncthreads();
  return total;
}

__device__ __forceinline__ uint32_t score_key(float v) {        // v >= 0 -> bits; invalid (< 0) -> 0
  return v > 0.f ? __float_as_uint(v) : 0u;
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
  float *sigma_out;         // scan's position scores [B][sigma_stride]
  int64_t sigma_stride;
  int32_t *d_err;
  int32_t use_pool;         // position stage reads pool_in instead of the candidate list
  const int32_t *row_seq;   // verify rows: [rows] session of each query row (null: one row per sequence)
  const int64_t *row_pos;   // verify rows: [rows] position of each query row (causal limit)
};

// One unit of the position stage: a sequence, or (verify rows) one query row of a session.
// q, w, workspace slices and outputs are indexed by r; the pool and the keys by b; positions
// at or beyond e.len are not candidates (the causal limit of a verify row); nb_seq counts the
// whole sequence's blocks (pool ids beyond it are errors).
struct SelUnit {
  int r, b;
  SeqTable e;
  int64_t nb_seq;
};

template <int BLOCK>
__device__ __forceinline__ SelUnit sel_unit(const IdxArgs &a, int r) {
  SelUnit u;
  u.r = r;
  if (!a.row_seq) {
    u.b = r;
    u.e = seq_entry(a.c, r, a.max_len, nullptr);
    u.nb_seq = (u.e.len + BLOCK - 1) / BLOCK;
    return u;
  }
  const int b = a.row_seq[r];
  const int64_t p = a.row_pos[r];
  if (b < 0 || b >= a.c.B) {
    if (threadIdx.x == 0) set_err(a.d_err, CSA2_DEVERR_SEQ);
    u.b = 0;
    u.e.len = 0;
    u.e.base = 0;
    u.nb_seq = 0;
    return u;
  }
  u.b = b;
  u.e = seq_entry(a.c, b, a.max_len, nullptr);
  u.nb_seq = (u.e.len + BLOCK - 1) / BLOCK;
  if (p < 0 || p >= u.e.len) {
    if (threadIdx.x == 0) set_err(a.d_err, CSA2_DEVERR_POS);
    u.e.len = 0;
  } else {
    u.e.len = (int32_t)(p + 1);
  }
  return u;
}

// ------------------------------------------------------------------ scan

// One CTA of 16 warps per SM: measured on B300, co-resident CTAs of the same kernel progress
// unevenly (the last-started CTA of each SM finished ~3 us after the first at 64K context),
// which a single CTA per SM avoids.
#ifndef CSA2_SCAN_WARPS
#define CSA2_SCAN_WARPS 16
#endif
#ifndef CSA2_SCAN_STAGES
#define CSA2_SCAN_STAGES 4
#endif
#ifndef CSA2_SCAN_CTAS
#define CSA2_SCAN_CTAS 1
#endif
constexpr int kScanWarps = CSA2_SCAN_WARPS;
constexpr int kScanStages = CSA2_SCAN_STAGES;
constexpr int kStageRows = 32;
constexpr int kStageBytes = kStageRows * kDIdx + kStageRows * 4;   // 2,176 B
constexpr int kScanSmemPerWarp = kScanStages * kStageBytes;
constexpr int kScanSmem = kScanWarps * kScanSmemPerWarp;


// four E4M3 codes -> two f16x2 (bytes 0,1 -> lo; bytes 2,3 -> hi), exact
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Scores of a 32-row stage held as rows g, g+8 (tile A) and g+16, g+24 (tile B).  The quad partial sums are combined with a butterfly transpose-reduce
// (3 shuffles instead of 8) so that lane t of each quad ends with row set t: the returned
// value is the score of stage row 8t + g.
__device__ __forceinline__ float score32_row(const QFrag &f, const uint4 &ka, const uint4 &ka8, const uint4 &kb,
                                            const uint4 &kb8, const float4 &s, int t) {
  float ca[4] = {0.f, 0.f, 0.f, 0.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wa8[4] = {ka8.x, ka8.y, ka8.z, ka8.w};
  const uint32_t wb[4] = {kb.x, kb.y, kb.z, kb.w}, wb8[4] = {kb8.x, kb8.y, kb8.z, kb8.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t a0, a2, a1, a3, b0, b2, b1, b3;
    e4m3x4_to_f16x4(wa[j], a0, a2);
    e4m3x4_to_f16x4(wa8[j], a1, a3);
    e4m3x4_to_f16x4(wb[j], b0, b2);
    e4m3x4_to_f16x4(wb8[j], b1, b3);
    mma_16816(ca, a0, a1, a2, a3, f.b[j][0], f.b[j][1]);
    mma_16816(cb, b0, b1, b2, b3, f.b[j][0], f.b[j][1]);
  }
  const float p0 = fmaxf(ca[0], 0.f) * f.wi0 + fmaxf(ca[1], 0.f) * f.wi1;   // row set 0: rows g
  const float p1 = fmaxf(ca[2], 0.f) * f.wi0 + fmaxf(ca[3], 0.f) * f.wi1;   // row set 1: rows g+8
  const float p2 = fmaxf(cb[0], 0.f) * f.wi0 + fmaxf(cb[1], 0.f) * f.wi1;   // row set 2: rows g+16
  const float p3 = fmaxf(cb[2], 0.f) * f.wi0 + fmaxf(cb[3], 0.f) * f.wi1;   // row set 3: rows g+24
  const bool b0 = t & 1, b1 = t & 2;
  const float r1 = __shfl_xor_sync(0xffffffffu, b0 ? p0 : p1, 1);
  const float r2 = __shfl_xor_sync(0xffffffffu, b0 ? p2 : p3, 1);
  const float sa = (b0 ? p1 : p0) + r1;                                       // set b0 (pair sum)
  const float sb = (b0 ? p3 : p2) + r2;                                       // set 2 + b0
  const float r3 = __shfl_xor_sync(0xffffffffu, b1 ? sa : sb, 2);
  const float tot = (b1 ? sb : sa) + r3;                                      // set t, whole quad
  const float sc = t == 0 ? s.x : t == 1 ? s.y : t == 2 ? s.z : s.w;
  const float o = tot * sc;
  return o > 0.f ? o : 0.f;                                                   // also maps NaN and -0 to +0
}

// Block maxima of one stage from per-lane row scores (lane (g, t) holds stage row 8t+g):
// xor-shuffles over the lanes of each block (uniform across the warp), then the block's
// first lane writes it and counts it in the histogram (the CTA's shared copy for its home
// sequence, else the global one).  `rows`: valid rows of the stage; blk0: the stage's
// first block id within the sequence.
template <int BLOCK>
__device__ __forceinline__ void emit_stage(float o, int lane, int blk0, int rows, float *bmax, uint32_t *s_hist,
                                           uint32_t *g_hist, bool home) {
  const int g = lane >> 2, t = lane & 3;
  float m = o;
#pragma unroll
  for (int s = 4; s < 4 * (BLOCK < 8 ? BLOCK : 8); s <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
  if constexpr (BLOCK == 16) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  const int row = 8 * t + g;
  const bool writer = BLOCK == 16 ? (g == 0 && (t & 1) == 0) : (g % BLOCK) == 0;
  if (writer && row < rows) {
    bmax[blk0 + row / BLOCK] = m;
    const uint32_t bin = min(__float_as_uint(m) >> kHistShift, (uint32_t)kHistBins - 1);
    if (home) atomicAdd(&s_hist[bin], 1u);
    else atomicAdd(&g_hist[bin], 1u);
  }
}

// Each warp streams a contiguous range of 32-row stages through its own ring in shared
// memory (kScanStages stages), so loads in flight hold no registers: a stage's key rows
// arrive by one TMA bulk copy (issued by lane 0, completing the slot's mbarrier by byte
// count), its scales by one 4-byte cp.async per lane.  Stages never straddle sequences:
// sequence b has ceil(len_b / 32) of them and the warps split the concatenated list evenly.
// Stage layout: 32 rows x 64 key bytes, then 32 scales stored so that lane quad g finds
// rows g, g+8, g+16, g+24 in one 16-byte word.  Rows past the sequence's end get scale 0
// (their keys are whatever follows in the cache, or stale), so they score 0.
template <int BLOCK, bool SIGMA, bool PRIV>
__global__ void __launch_bounds__(kScanWarps * 32, CSA2_SCAN_CTAS)
    scan_kernel(const __grid_constant__ IdxArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) uint8_t s_dyn[];
  __shared__ __align__(8) uint64_t s_full[kScanWarps][kScanStages];     // key rows of each ring slot
  static_assert((kScanStages & (kScanStages - 1)) == 0, "ring length must be a power of two");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (lane == 0) {
    for (int i = 0; i < kScanStages; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_addr(&s_full[warp][i])));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncwarp();
  const int B = a.c.B;
  uint32_t *s_hist = reinterpret_cast<uint32_t *>(s_dyn + kScanSmem);   // PRIV: [kHistBins] home sequence's counts
  int64_t *s_first = reinterpret_cast<int64_t *>(s_hist + (PRIV ? kHistBins : 0));   // [B + 1] first stage of each sequence
  int64_t *s_base = s_first + (B + 1);
  int32_t *s_len = reinterpret_cast<int32_t *>(s_base + B);
  for (int i = tid; i < B; i += blockDim.x) {
    SeqTable e = seq_entry(a.c, i, a.max_len, blockIdx.x == 0 ? a.d_err : nullptr);
    s_len[i] = e.len;
    s_base[i] = e.base;
  }
  if (PRIV)
    for (int i = tid; i < kHistBins; i += blockDim.x) s_hist[i] = 0u;
  __syncthreads();
  if (warp == 0) {   // exclusive prefix of stages per sequence
    const int per = (B + 31) / 32;
    int64_t local = 0;
    for (int i = lane * per; i < min(B, lane * per + per); ++i) local += (s_len[i] + 31) / 32;
    int64_t incl = local;
    for (int o = 1; o < 32; o <<= 1) {
      int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int64_t run = incl - local;
    for (int i = lane * per; i < min(B, lane * per + per); ++i) { s_first[i] = run; run += (s_len[i] + 31) / 32; }
    if (lane == 31) s_first[B] = incl;
  }
  __syncthreads();
  const int64_t total = s_first[B];
  const int64_t W = (int64_t)gridDim.x * kScanWarps;
  const int64_t gw = (int64_t)blockIdx.x * kScanWarps + warp;
  const int64_t g_begin = total * gw / W, g_end = total * (gw + 1) / W;
  const int nst = (int)(g_end - g_begin);
  const int g = lane >> 2, t = lane & 3;
  // sequence holding global stage x (skipping empty sequences); x < total
  auto seq_of = [&](int64_t x) {
    int lo = 0, hi = B;                                          // s_first[lo] <= x < s_first[hi]
    while (hi - lo > 1) { int mid = (lo + hi) >> 1; if (s_first[mid] <= x) lo = mid; else hi = mid; }
    while (s_first[lo + 1] == s_first[lo]) ++lo;
    return lo;
  };
  const int64_t cta_first = total * ((int64_t)blockIdx.x * kScanWarps) / W;
  const int home_b = PRIV && cta_first < total ? seq_of(cta_first) : -1;  // the CTA's shared histogram counts this one
  if (nst > 0) {
  const int b0 = seq_of(g_begin);
  uint8_t *ring = s_dyn + warp * kScanSmemPerWarp;
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
  const uint32_t sc_dst = kStageRows * kDIdx + 4 * ((lane & 7) * 4 + (lane >> 3));

  // producer cursor: sequence, stage within it, its stage count and length, first row
  int pb = b0, ps = (int)(g_begin - s_first[b0]);
  int pn = (int)(s_first[b0 + 1] - s_first[b0]), plen = s_len[b0];
  int64_t prow = s_base[b0] + 32 * (int64_t)ps;
  // issue the loads of this warp's next stage into ring slot k
  auto issue_stage = [&](int k) {
    if (ps == pn) {                                              // next sequence with stages
      do { ++pb; } while (s_first[pb + 1] == s_first[pb]);
      ps = 0;
      pn = (int)(s_first[pb + 1] - s_first[pb]);
      plen = s_len[pb];
      prow = s_base[pb];
    }
    const int slot = k & (kScanStages - 1);
    const uint32_t dst = ring_s + (uint32_t)slot * kStageBytes;
    const int rows = min(32, plen - 32 * ps);
    if (lane == 0) {                                             // key rows that exist in the cache
      const int64_t avail = a.c.T_cap - prow;
      const uint32_t bytes = (uint32_t)(avail < kStageRows ? avail : kStageRows) * kDIdx;
      fence_async_smem();                                        // the slot's last reads precede the copy
      mbar_expect_tx_u32(smem_addr(&s_full[warp][slot]), bytes);
      bulk_copy_g2s(dst, a.c.ik_codes + prow * kDIdx, bytes, smem_addr(&s_full[warp][slot]));
    }
    cp_async4(dst + sc_dst, lane < rows ? a.c.ik_scale + prow + lane : a.c.ik_scale, lane < rows);
    cp_async_commit();
    ++ps;
    prow += kStageRows;
  };
  const int pre = min(kScanStages - 1, nst);
  for (int s = 0; s < pre; ++s) issue_stage(s);
  for (int s = pre; s < kScanStages - 1; ++s) cp_async_commit();

  // consumer cursor mirrors the producer
  int cb = b0, cs = (int)(g_begin - s_first[b0]);
  int cn = (int)(s_first[b0 + 1] - s_first[b0]), clen = s_len[b0];
  QFrag f;
  load_qfrag(a.q + (int64_t)cb * kHIdx * kDIdx, a.w + (int64_t)cb * kHIdx, lane, f);
  float smx = 0.f;
  float *bmax = a.ws.bmax + (int64_t)cb * a.ws.nbm;
  uint32_t *hist = a.ws.hist + (int64_t)cb * kHistBins;
  bool home = cb == home_b;
  auto consume = [&](int k) {
    const bool landed = mbar_wait_spin(smem_addr(&s_full[warp][k & (kScanStages - 1)]), (k / kScanStages) & 1);
    if (!landed && lane == 0) set_err(a.d_err, CSA2_DEVERR_TIMEOUT);
    cp_async_wait<kScanStages - 1>();
    __syncwarp();
    if (cs == cn) {                                              // a new sequence: its queries and weights
      const float m = warp_max(smx);
      if (lane == 0 && m > 0.f) atomicMax(&a.ws.smax[cb], __float_as_uint(m));
      do { ++cb; } while (s_first[cb + 1] == s_first[cb]);
      cs = 0;
      cn = (int)(s_first[cb + 1] - s_first[cb]);
      clen = s_len[cb];
      load_qfrag(a.q + (int64_t)cb * kHIdx * kDIdx, a.w + (int64_t)cb * kHIdx, lane, f);
      smx = 0.f;
      bmax = a.ws.bmax + (int64_t)cb * a.ws.nbm;
      hist = a.ws.hist + (int64_t)cb * kHistBins;
      home = cb == home_b;
    }
    const uint8_t *st = ring + (k & (kScanStages - 1)) * kStageBytes;
    const uint4 ka = *reinterpret_cast<const uint4 *>(st + g * kDIdx + 16 * t);
    const uint4 ka8 = *reinterpret_cast<const uint4 *>(st + (g + 8) * kDIdx + 16 * t);
    const uint4 kb = *reinterpret_cast<const uint4 *>(st + (g + 16) * kDIdx + 16 * t);
    const uint4 kb8 = *reinterpret_cast<const uint4 *>(st + (g + 24) * kDIdx + 16 * t);
    const float4 sc = *reinterpret_cast<const float4 *>(st + kStageRows * kDIdx + 16 * g);
    __syncwarp();
    const float o = score32_row(f, ka, ka8, kb, kb8, sc, t);
    smx = fmaxf(smx, fmaxf(fmaxf(sc.x, sc.y), fmaxf(sc.z, sc.w)));
    const int rows = min(32, clen - 32 * cs);
    if (SIGMA) {
      const int row = 8 * t + g;
      if (row < rows) a.sigma_out[(int64_t)cb * a.sigma_stride + 32 * cs + row] = o;
    }
    emit_stage<BLOCK>(o, lane, 32 / BLOCK * cs, rows, bmax, s_hist, hist, home);
    ++cs;
  };
  // steady state: every iteration issues one stage and consumes one; then the ring drains
  int k = 0;
#pragma unroll 2
  for (; k + kScanStages - 1 < nst; ++k) {
    issue_stage(k + kScanStages - 1);
    consume(k);
  }
  for (; k < nst; ++k) {
    cp_async_commit();
    consume(k);
  }
  cp_async_wait<0>();
  const float m = warp_max(smx);
  if (lane == 0 && m > 0.f) atomicMax(&a.ws.smax[cb], __float_as_uint(m));
  }
  // the home sequence's counts join the global histogram
  if (PRIV) __syncthreads();
  if (PRIV && home_b >= 0) {
    uint32_t *gh = a.ws.hist + (int64_t)home_b * kHistBins;
    for (int i = tid; i < kHistBins; i += blockDim.x) {
      const uint32_t c = s_hist[i];
      if (c) atomicAdd(&gh[i], c);
    }
  }
}

// ------------------------------------------------------------------ candidate collection

constexpr int kCollectPer = 4096;   // block maxima per CTA

// Lower edge of the histogram bin holding the k-th largest block maximum.  Needs a
// 256-thread CTA: thread t sums the 16 bins [4096-16(t+1), 4096-16t) (top-down order),
// a CTA scan finds the chunk that crosses k, and its owner walks the 16 bins.
__device__ float hist_threshold_low(const uint32_t *hist_g, int k, int *s_scan, int *s_misc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint4 *src = reinterpret_cast<const uint4 *>(hist_g + kHistBins - 16 * (tid + 1));
  uint32_t bins[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = __ldcg(src + j);
    bins[4 * j] = v.x; bins[4 * j + 1] = v.y; bins[4 * j + 2] = v.z; bins[4 * j + 3] = v.w;
  }
  int sum = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) sum += (int)bins[j];
  int incl = sum;
  for (int o = 1; o < 32; o <<= 1) { int v = __shfl_up_sync(0xffffffffu, incl, o); if (lane >= o) incl += v; }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += s_scan[w];
  incl += before;
  int excl = incl - sum;
  if (excl < k && k <= incl) {
    for (int j = 15; j >= 0; --j) {       // bins of this chunk from the top down
      excl += (int)bins[j];
      if (excl >= k) { s_misc[0] = kHistBins - 16 * (tid + 1) + j; break; }
    }
  }
  __syncthreads();
  const float th = __uint_as_float((uint32_t)s_misc[0] << kHistShift);
  __syncthreads();
  return th;
}

template <int BLOCK>
__global__ void __launch_bounds__(256) collect_kernel(const __grid_constant__ IdxArgs a) {
  pdl_enter();
  constexpr int kPer = kCollectPer / 256;
  __shared__ int s_scan[8];
  __shared__ int s_misc[4];
  __shared__ float s_E;
  __shared__ uint32_t s_base;
  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const SeqTable e = seq_entry(a.c, b, a.max_len, nullptr);
  const int64_t nb = (e.len + BLOCK - 1) / BLOCK;
  const int64_t j0 = (int64_t)blockIdx.x * kCollectPer;
  if (j0 >= nb) return;
  const int64_t j1 = min(nb, j0 + kCollectPer);
  const float *bm = a.ws.bmax + (int64_t)b * a.ws.nbm;
  float v[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {           // all loads in flight before the threshold work
    const int64_t j = j0 + k * 256 + tid;
    v[k] = j < j1 ? __ldcg(bm + j) : -FLT_MAX;
  }
  float thr = -FLT_MAX;
  if (nb > a.n_keep) {
    if (tid < 32) {
      const float E = seq_bound(a.q + (int64_t)b * kHIdx * kDIdx, a.w + (int64_t)b * kHIdx,
                                __uint_as_float(a.ws.smax[b]), tid);
      if (tid == 0) s_E = E;
    }
    const float th_low = hist_threshold_low(a.ws.hist + (int64_t)b * kHistBins, a.n_keep, s_scan, s_misc);
    thr = lo_cut(th_low, s_E);
  }
  int cnt = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) cnt += (j0 + k * 256 + tid < j1 && v[k] >= thr);
  int incl = cnt;
  for (int o = 1; o < 32; o <<= 1) { int x = __shfl_up_sync(0xffffffffu, incl, o); if (lane >= o) incl += x; }
  __syncthreads();
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
  for (int w = 0; w < 8; ++w) { total += s_scan[w]; if (w < warp) before += s_scan[w]; }
  if (tid == 0) s_base = total ? atomicAdd(&a.ws.cand_cnt[b], (uint32_t)total) : 0u;
  __syncthreads();
  uint64_t *cand = a.ws.cand + (int64_t)b * a.ws.nbm;
  uint32_t off = s_base + before + incl - cnt;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int64_t j = j0 + k * 256 + tid;
    if (j < j1 && v[k] >= thr) cand[off++] = ((uint64_t)__float_as_uint(v[k]) << 32) | (uint32_t)j;
  }
}

// ------------------------------------------------------------------ selection

// One CTA per sequence selects from items (block maxima or position scores):
//   1. the histogram of the items' float bits (4096 bins, built by the kernel that scored
//      them) gives the bin of the k-th largest approximate value;
//   2. one pass over the staged items, a warp per 32-item word, marks the items that are
//      certainly in (above the upper cut of the bin's upper edge) with ballots and counts
//      the items near the bin (between the cuts of its edges); a second pass lists them;
//   3. a radix selection over that list gives the exact k-th approximate value, whose cuts
//      split the list into certainly in, certainly out and the band;
//   4. band items are rescored exactly and ranked by (exact score desc, id asc).
#ifndef CSA2_SEL_THREADS
#define CSA2_SEL_THREADS 512
#endif
constexpr int kSelCta = CSA2_SEL_THREADS;
constexpr int kSelWarps = kSelCta / 32;
constexpr int kDirectBlocks = 16384;         // up to this many blocks a sequence's maxima are read directly
constexpr int kStageItems = 16384;           // items staged in shared memory
constexpr int kListCap = 2048;               // near-threshold items kept in shared memory
constexpr int kIdWords = 4096;               // block-id bitmaps: 131,072 blocks
constexpr int kItemWords = kMaxSel * 16 / 32;   // position-item bitmap: 65,536 items
static_assert(kHistBins % kSelCta == 0, "histogram bins per thread");

__device__ __forceinline__ float bin_lo(uint32_t bin) { return __uint_as_float(bin << kHistShift); }
__device__ __forceinline__ float bin_hi(uint32_t bin) { return __uint_as_float((bin + 1u) << kHistShift); }

// Top-down bins of the ka-th and kb-th largest (1-based; a k outside [1, total] is not
// looked for) over kHistBins counts.  s_out = {bin_a, above_a, bin_b, above_b, total}.
// Needs blockDim.x == kSelCta.
template <class CountFn>
__device__ void cta_find_bins(int ka, int kb, CountFn count, int *s_scan, int *s_out) {
  constexpr int PER = kHistBins / kSelCta;
  const int top = kHistBins - 1 - (int)threadIdx.x * PER;         // this thread's highest bin
  int c[PER];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) { c[i] = (int)count(top - i); sum += c[i]; }
  const int excl = cta_excl_scan(sum, s_scan);
  if (threadIdx.x == 0) s_out[4] = s_scan[64];
  if (excl < ka && ka <= excl + sum) {
    int run = excl;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if (run + c[i] >= ka) { s_out[0] = top - i; s_out[1] = run; break; }
      run += c[i];
    }
  }
  if (excl < kb && kb <= excl + sum) {
    int run = excl;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if (run + c[i] >= kb) { s_out[2] = top - i; s_out[3] = run; break; }
      run += c[i];
    }
  }
  __syncthreads();
}

// r-th largest key (1 <= r <= matching items) among list entries, whose keys minus `base`
// lie in [0, range]: radix passes of up to 11 bits over the list only.
template <class KeyFn>
__device__ uint32_t list_kth(const int32_t *m, int cnt, KeyFn key, int r, uint32_t base, uint32_t range,
                             uint32_t *s_hist, int *s_scan, int *s_out) {
  const int tid = threadIdx.x;
  int shift = range ? 32 - __clz((int)range) : 0;
  uint32_t prefix = 0;
  while (shift > 0) {
    const int w = min(11, shift);
    const int sub = shift - w;
    const int nbins = 1 << w;
    for (int i = tid; i < nbins; i += blockDim.x) s_hist[i] = 0u;
    __syncthreads();
    for (int j = tid; j < cnt; j += blockDim.x) {
      const uint32_t d = key(m[j]) - base;
      const bool match = shift >= 32 || (d >> shift) == prefix;
      if (match) atomicAdd(&s_hist[(d >> sub) & (uint32_t)(nbins - 1)], 1u);
    }
    __syncthreads();
    cta_find_bin(nbins, r, [&](int bb) { return s_hist[bb]; }, s_scan, s_out);
    prefix = (prefix << w) | (uint32_t)s_out[0];
    r -= s_out[1];
    shift = sub;
  }
  return base + prefix;
}

// Marks the top `need` band entries by (exact score desc, id asc); a warp per entry.
template <class IdFn, class PickFn>
__device__ void rank_band(const int32_t *band, const float2 *ex, int u, int need, IdFn id, PickFn pick) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int i = warp; i < u; i += nwarps) {
    const float2 vi = ex[i];
    const int32_t ii = id(band[i]);
    int rank = 0;
    for (int m = lane; m < u; m += 32) {
      const float2 vm = ex[m];
      rank += df_greater(vm, vi) || (df_equal(vm, vi) && id(band[m]) < ii);
    }
    rank = __reduce_add_sync(0xffffffffu, rank);
    if (lane == 0 && rank < need) pick(band[i]);
  }
}

// Exact maxima of band blocks, one warp per block.  The block's rows are first scored on
// the tensor cores; only rows whose upper bound reaches the best lower bound of the block
// are rescored exactly (usually one).
template <int BLOCK, class IdFn>
__device__ void exact_block_maxima(const IdxArgs &a, const SeqTable &e, const QFrag &f, const QExact &q, float E,
                                   const int32_t *band, float2 *ex, int u, IdFn id, const int32_t *lut) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const float up = 1.0f + 2.0f * kRelF, dn = 1.0f - 2.0f * kRelF;
  for (int i = warp; i < u; i += nwarps) {
    const int32_t j = id(band[i]);
    const int rg = g, rg8 = g + 8;
    const int64_t p0 = (int64_t)j * BLOCK + rg, p8 = (int64_t)j * BLOCK + rg8;
    const bool v0 = rg < BLOCK && p0 < e.len, v8 = rg8 < BLOCK && p8 < e.len;
    const uint4 k0 = v0 ? ld_nc16(a.c.ik_codes + (e.base + p0) * kDIdx + 16 * t) : make_uint4(0, 0, 0, 0);
    const uint4 k8 = v8 ? ld_nc16(a.c.ik_codes + (e.base + p8) * kDIdx + 16 * t) : make_uint4(0, 0, 0, 0);
    const float s0 = v0 ? __ldg(a.c.ik_scale + e.base + p0) : 0.f;
    const float s8 = v8 ? __ldg(a.c.ik_scale + e.base + p8) : 0.f;
    float o0, o8;
    score16(f, k0, k8, s0, s8, o0, o8);
    const float lo0 = v0 ? __fsub_rd(__fmul_rd(dn, o0), E) : -FLT_MAX;
    const float lo8 = v8 ? __fsub_rd(__fmul_rd(dn, o8), E) : -FLT_MAX;
    const float best_lo = fmaxf(0.f, warp_max(fmaxf(lo0, lo8)));
    const float hi0 = __fadd_ru(__fmul_ru(up, o0), E), hi8 = __fadd_ru(__fmul_ru(up, o8), E);
    // rows that can still be the block's maximum
    unsigned cand = __ballot_sync(0xffffffffu, t == 0 && v0 && hi0 >= best_lo);
    unsigned cand8 = __ballot_sync(0xffffffffu, t == 0 && v8 && hi8 >= best_lo);
    float2 best = make_float2(-1.f, 0.f);
    while (cand | cand8) {
      const bool from8 = cand == 0u;
      const int src = __ffs(from8 ? cand8 : cand) - 1;          // lane t = 0 of the row's quad
      if (from8) cand8 &= cand8 - 1; else cand &= cand - 1;
      const uint4 kk = make_uint4(__shfl_sync(0xffffffffu, from8 ? k8.x : k0.x, src + t),
                                  __shfl_sync(0xffffffffu, from8 ? k8.y : k0.y, src + t),
                                  __shfl_sync(0xffffffffu, from8 ? k8.z : k0.z, src + t),
                                  __shfl_sync(0xffffffffu, from8 ? k8.w : k0.w, src + t));
      const float ss = __shfl_sync(0xffffffffu, from8 ? s8 : s0, src);
      const float2 v = exact_sigma(q, kk, ss, lut);
      if (df_greater(v, best)) best = v;
    }
    if (lane == 0) ex[i] = best;
  }
}

enum { kCntIn = 0, kCntBand = 1, kCntPcb = 2, kCntSort = 3 };

// Steps 3-4 for one threshold: exact k-th approximate value among the listed items, then
// marks (via pick) the listed items that belong to the top k.  Every thread calls it.
// `m`/`mc`: the near list; n_cert items above it are already marked.
template <class ValFn, class IdFn, class ExactFn, class PickFn>
__device__ void resolve_list(const int32_t *m, int mc, int k, int n_cert, float w_lo, float w_hi, float E, ValFn val,
                             IdFn id, ExactFn exact_band, PickFn pick, int32_t *band, float2 *ex, uint32_t *s_hist,
                             int *s_cnt, int *s_scan, int *s_out) {
  const int r = k - n_cert;
  const uint32_t kth = list_kth(m, mc, [&](int i) { return __float_as_uint(val(i)); }, r, __float_as_uint(w_lo),
                                __float_as_uint(w_hi) - __float_as_uint(w_lo), s_hist, s_scan, s_out);
  const float theta = __uint_as_float(kth);
  const float hi = hi_cut(theta, E), lo = lo_cut(theta, E);
  if (threadIdx.x == 0) { s_cnt[kCntIn] = 0; s_cnt[kCntBand] = 0; }
  __syncthreads();
  const int iters = (mc + blockDim.x - 1) / blockDim.x;
  for (int it = 0; it < iters; ++it) {
    const int j = it * blockDim.x + threadIdx.x;
    const int i = j < mc ? m[j] : 0;
    const float v = j < mc ? val(i) : -1.f;
    const bool in = j < mc && v > hi;
    const bool bd = j < mc && !in && v >= lo;
    if (warp_reserve(in, &s_cnt[kCntIn]) >= 0) pick(i);
    const int s = warp_reserve(bd, &s_cnt[kCntBand]);
    if (bd) band[s] = i;
  }
  __syncthreads();
  const int n_in = s_cnt[kCntIn], u = s_cnt[kCntBand];
  if (u > 0) exact_band(band, ex, u);
  __syncthreads();
  rank_band(band, ex, u, r - n_in, id, pick);
}

// Warp-per-word classification of items [0, n) against up to two thresholds (a, b): each
// 32-item word's "certain" ballot goes to cert_word(w, bits) (or to pick one by one), the
// "near" items are counted per warp and then listed in item order.  Returns nothing; the
// lists and counts are left in m_a / m_b and s_tot = {near_a, near_b, cert_a, cert_b}.
struct NearLists {
  int32_t *sa, *sb;      // shared lists (kListCap)
  int32_t *ga, *gb;      // global lists (used when a list exceeds kListCap)
};
template <class ValFn, class CertFn>
__device__ void classify_words(int n, ValFn val, bool use_a, float a_lo, float a_hi, bool use_b, float b_lo,
                               float b_hi, CertFn cert, const NearLists &L, int (*s_wc)[4], int *s_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int nw = (n + 31) / 32;
  int na = 0, nbb = 0, ca = 0, cb = 0;
  for (int w = warp; w < nw; w += nwarps) {
    const int i = 32 * w + lane;
    const float v = i < n ? val(i) : -1.f;
    const bool ok = v >= 0.f;
    const unsigned c1 = __ballot_sync(0xffffffffu, use_a && ok && v > a_hi);
    const unsigned n1 = __ballot_sync(0xffffffffu, use_a && ok && v <= a_hi && v >= a_lo);
    const unsigned c2 = __ballot_sync(0xffffffffu, use_b && ok && v > b_hi);
    const unsigned n2 = __ballot_sync(0xffffffffu, use_b && ok && v <= b_hi && v >= b_lo);
    cert(w, i, c1, c2);
    na += __popc(n1); nbb += __popc(n2); ca += __popc(c1); cb += __popc(c2);
  }
  if (lane == 0) { s_wc[warp][0] = na; s_wc[warp][1] = nbb; s_wc[warp][2] = ca; s_wc[warp][3] = cb; }
  __syncthreads();
  int oa = 0, ob = 0, ta = 0, tb = 0, tca = 0, tcb = 0;
  for (int x = 0; x < nwarps; ++x) {
    if (x < warp) { oa += s_wc[x][0]; ob += s_wc[x][1]; }
    ta += s_wc[x][0]; tb += s_wc[x][1]; tca += s_wc[x][2]; tcb += s_wc[x][3];
  }
  if (threadIdx.x == 0) { s_tot[0] = ta; s_tot[1] = tb; s_tot[2] = tca; s_tot[3] = tcb; }
  int32_t *la = ta <= kListCap ? L.sa : L.ga;
  int32_t *lb = tb <= kListCap ? L.sb : L.gb;
  const unsigned lt = (1u << lane) - 1u;
  for (int w = warp; w < nw; w += nwarps) {
    const int i = 32 * w + lane;
    const float v = i < n ? val(i) : -1.f;
    const bool ok = v >= 0.f;
    const bool in_a = use_a && ok && v <= a_hi && v >= a_lo;
    const bool in_b = use_b && ok && v <= b_hi && v >= b_lo;
    const unsigned n1 = __ballot_sync(0xffffffffu, in_a);
    const unsigned n2 = __ballot_sync(0xffffffffu, in_b);
    if (in_a) la[oa + __popc(n1 & lt)] = i;
    if (in_b) lb[ob + __popc(n2 & lt)] = i;
    oa += __popc(n1);
    ob += __popc(n2);
  }
  __syncthreads();
}

// Approximate scores of the positions of an ascending block list (units of 16 positions;
// this warp takes units u_first, u_first + u_step, ...; the loads of four units are issued
// before any arithmetic).  Invalid positions score -1; valid ones are also counted in the
// sequence's score histogram.
template <int BLOCK>
__device__ void score_units(const IdxArgs &a, const SeqTable &e, int64_t nb, const int32_t *list, int n, float *pv,
                            uint32_t *hist, const QFrag &f, int u_first, int u_step, float &smx) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int units = (n + 15) / 16;
  for (int u0 = u_first; u0 < units; u0 += 4 * u_step) {
    uint4 k[4][2];
    float s[4][2];
    bool ok[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = (u0 + j * u_step) * 16 + g + 8 * h;
        int64_t p = -1;
        if (u0 + j * u_step < units && i < n) {
          const int32_t blk = list[i / BLOCK];
          if (blk >= 0) {
            if (blk >= nb) {
              if (t == 0) set_err(a.d_err, CSA2_DEVERR_POOL);
            } else {
              p = (int64_t)blk * BLOCK + (i % BLOCK);
              if (p >= e.len) p = -1;
            }
          }
        }
        ok[j][h] = p >= 0;
        const int64_t row = e.base + (p >= 0 ? p : 0);
        k[j][h] = p >= 0 ? ld_nc16(a.c.ik_codes + row * kDIdx + 16 * t) : make_uint4(0, 0, 0, 0);
        s[j][h] = p >= 0 ? __ldg(a.c.ik_scale + row) : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (u0 + j * u_step >= units) break;
      float o[2];
      score16(f, k[j][0], k[j][1], s[j][0], s[j][1], o[0], o[1]);
      smx = fmaxf(smx, fmaxf(s[j][0], s[j][1]));
      if (t == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = (u0 + j * u_step) * 16 + g + 8 * h;
          if (i < n) {
            pv[i] = ok[j][h] ? o[h] : -1.f;
            if (ok[j][h]) atomicAdd(&hist[min(__float_as_uint(o[h]) >> kHistShift, (uint32_t)kHistBins - 1)], 1u);
          }
        }
      }
    }
  }
}

// Shared tail of the position selections: items [0, n) with approximate scores val(i)
// (-1 invalid), n_valid of them valid, the topk-th largest in histogram bin `bin`.
// Writes the exact top-k positions ascending to out (-1 padded).  Every thread calls it.
struct PosWork {
  uint32_t *radix;     // [2048] radix scratch
  uint32_t *bits;      // item bitmap, ceil(n / 32) words
  int32_t *m, *band;   // [kListCap]
  float2 *ex;          // [kListCap]
  const int32_t *lut;  // [256]
  int *cnt, *scan, *out;
  int (*wc)[4];
  int *tot;
};

template <int BLOCK, class ValFn, class PosFn>
__device__ void select_positions_core(const IdxArgs &a, const SeqTable &e, int b, int n, int n_valid, uint32_t bin,
                                      ValFn val, PosFn pos_of, float E, const PosWork &w, int32_t *out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint16_t *qb = a.q + (int64_t)b * kHIdx * kDIdx;
  const float *wb = a.w + (int64_t)b * kHIdx;
  auto id = [](int i) -> int32_t { return i; };                      // item order = position order
  auto pick = [&](int i) { atomicOr(&w.bits[i >> 5], 1u << (i & 31)); };
  auto cert = [&](int word, int, unsigned c1, unsigned) { if (lane == 0) w.bits[word] = c1; };
  int32_t *g_m = a.ws.unc_id + (int64_t)b * 3 * a.ws.unc_x;
  if (n_valid <= a.topk) {
    // every valid score is selected: "certain" = valid, nothing near
    classify_words(n, val, true, 1.f, -0.5f, false, 0.f, 0.f, cert, NearLists{w.m, w.m, g_m, g_m}, w.wc, w.tot);
  } else {
    const float w_hi = hi_cut(bin_hi(bin), E), w_lo = lo_cut(bin_lo(bin), E);
    classify_words(n, val, true, w_lo, w_hi, false, 0.f, 0.f, cert, NearLists{w.m, w.m, g_m, g_m}, w.wc, w.tot);
    const int mc = w.tot[0], n_cert = w.tot[2];
    const bool big = mc > kListCap;
    const int32_t *m = big ? g_m : w.m;
    int32_t *band = big ? g_m + a.ws.unc_x : w.band;
    float2 *ex = big ? a.ws.unc_val + (int64_t)b * a.ws.unc_x : w.ex;
    auto exact_band = [&](const int32_t *bd, float2 *xv, int u) {
      QExact q;
      load_qexact(qb, wb, lane, q);
      for (int j = warp; j < u; j += kSelWarps) {
        const int64_t row = e.base + pos_of(bd[j]);
        const uint4 kk = __ldg(reinterpret_cast<const uint4 *>(a.c.ik_codes + row * kDIdx + 16 * (lane & 3)));
        const float2 v = exact_sigma(q, kk, __ldg(a.c.ik_scale + row), w.lut);
        if (lane == 0) xv[j] = v;
      }
    };
    resolve_list(m, mc, a.topk, n_cert, w_lo, w_hi, E, val, id, exact_band, pick, band, ex, w.radix, w.cnt, w.scan,
                 w.out);
  }
  __syncthreads();
  emit_bits_ascending(w.bits, (n + 31) / 32, pos_of, out, a.topk, w.scan);
}

// ---- the Full layer after the scan: pool + position-candidate blocks

// The Full layer's selection after the scan, one CTA per sequence.
// Pool = the top min(n_keep, nb) blocks by (exact block score desc, id asc), ascending.
// Position-candidate blocks = every block whose approximate maximum reaches the lower cut
// of the topk-th largest approximate block maximum (they contain every top-k position);
// their positions, with the scores the scan stored, give the exact top-k positions.  DIRECT: the sequence's block maxima are the items (nb <= kDirectBlocks);
// otherwise the items are the candidates gathered by collect_kernel.  Both thresholds
// come from the scan's histogram of all block maxima.
template <int BLOCK, bool DIRECT>
__global__ void __launch_bounds__(kSelCta, 1) finalize_blocks_kernel(const __grid_constant__ IdxArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) uint8_t s_dyn[];
  uint32_t *s_hist = reinterpret_cast<uint32_t *>(s_dyn);            // radix scratch [2048]
  uint32_t *s_pool_bits = s_hist + 2048;
  uint32_t *s_pcb_bits = s_pool_bits + kIdWords;
  int32_t *s_m1 = reinterpret_cast<int32_t *>(s_pcb_bits + kIdWords);
  int32_t *s_m2 = s_m1 + kListCap;
  int32_t *s_band = s_m2 + kListCap;
  int32_t *s_band2 = s_band + kListCap;
  float2 *s_ex = reinterpret_cast<float2 *>(s_band2 + kListCap);
  int32_t *s_lut = reinterpret_cast<int32_t *>(s_ex + kListCap);
  float *s_val = reinterpret_cast<float *>(s_lut + 256);
  int32_t *s_id = reinterpret_cast<int32_t *>(s_val + kStageItems);  // candidate mode only
  __shared__ int s_cnt[8];
  __shared__ int s_scan[72];
  __shared__ int s_out[8];
  __shared__ int s_wc[kSelWarps][4];
  __shared__ int s_tot[4];
  __shared__ float s_E;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const SeqTable e = seq_entry(a.c, b, a.max_len, nullptr);
  const int nb = (int)((e.len + BLOCK - 1) / BLOCK);
  const int n_keep = a.n_keep;
  const int k1 = min(n_keep, nb), k2 = min(a.topk, nb);
  const bool sel_pool = nb > n_keep, sel_pcb = nb > a.topk;
  int32_t *pool = a.pool_out + (int64_t)b * n_keep;
  const uint16_t *qb = a.q + (int64_t)b * kHIdx * kDIdx;
  const float *wb = a.w + (int64_t)b * kHIdx;
  const uint32_t *hist_g = a.ws.hist + (int64_t)b * kHistBins;
  const uint64_t *cand_g = a.ws.cand + (int64_t)b * a.ws.nbm;
  const bool use_bits = nb <= kIdWords * 32;
  const int nwords = use_bits ? (nb + 31) / 32 : 0;

  if (!DIRECT)
    for (int i = tid; i < nwords; i += blockDim.x) { s_pool_bits[i] = 0u; s_pcb_bits[i] = 0u; }
  if (tid < 8) s_cnt[tid] = 0;
  fill_e4m3_lut(s_lut);
  if (warp == 0) {
    const float E = seq_bound(qb, wb, __uint_as_float(a.ws.smax[b]), lane);
    if (lane == 0) s_E = E;
  }
  // ---- stage the items
  int n;
  bool staged = true;
  if (DIRECT) {
    n = nb;
    const float *bm = a.ws.bmax + (int64_t)b * a.ws.nbm;            // 16-byte aligned rows
    const int n4 = n >> 2;
    for (int i = tid; i < n4; i += blockDim.x)
      reinterpret_cast<float4 *>(s_val)[i] = __ldcg(reinterpret_cast<const float4 *>(bm) + i);
    for (int i = 4 * n4 + tid; i < n; i += blockDim.x) s_val[i] = __ldcg(bm + i);
  } else {
    n = (int)a.ws.cand_cnt[b];
    staged = n <= kStageItems;
    if (staged) {
      const int n2 = n >> 1;
      for (int i = tid; i < n2; i += blockDim.x) {
        const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(cand_g) + i);
        s_val[2 * i] = __uint_as_float(v.y); s_id[2 * i] = (int32_t)v.x;
        s_val[2 * i + 1] = __uint_as_float(v.w); s_id[2 * i + 1] = (int32_t)v.z;
      }
      if ((n & 1) && tid == 0) {
        const uint64_t v = __ldcg(cand_g + n - 1);
        s_val[n - 1] = __uint_as_float((uint32_t)(v >> 32)); s_id[n - 1] = (int32_t)(uint32_t)v;
      }
    }
  }
  // ---- histogram bins of the k1-th and k2-th largest block maxima (syncs the staging)
  cta_find_bins(sel_pool ? k1 : 0, sel_pcb ? k2 : 0, [&](int bin) { return __ldcg(hist_g + bin); }, s_scan, s_out);
  const uint32_t bin1 = sel_pool ? (uint32_t)s_out[0] : 0u, bin2 = sel_pcb ? (uint32_t)s_out[2] : 0u;
  const float E = s_E;
  const float w1_hi = hi_cut(bin_hi(bin1), E), w1_lo = lo_cut(bin_lo(bin1), E);
  const float w2_hi = hi_cut(bin_hi(bin2), E), w2_lo = lo_cut(bin_lo(bin2), E);
  auto val = [&](int i) -> float {
    if (DIRECT || staged) return s_val[i];
    return __uint_as_float((uint32_t)(__ldcg(cand_g + i) >> 32));
  };
  auto id = [&](int i) -> int32_t {
    if (DIRECT) return i;
    if (staged) return s_id[i];
    return (int32_t)(uint32_t)__ldcg(cand_g + i);
  };
  // the sort buffer of the no-bitmap path reuses the pcb bitmap (pcb = pool there)
  int32_t *s_sort = reinterpret_cast<int32_t *>(s_pcb_bits);
  auto pick_pool = [&](int i) {
    const int32_t j = id(i);
    if (use_bits) atomicOr(&s_pool_bits[j >> 5], 1u << (j & 31));
    else s_sort[atomicAdd(&s_cnt[kCntSort], 1)] = j;
  };
  auto pick_pcb = [&](int i) {
    const int32_t j = id(i);
    if (use_bits) atomicOr(&s_pcb_bits[j >> 5], 1u << (j & 31));
  };
  auto cert = [&](int w, int i, unsigned c1, unsigned c2) {
    if (DIRECT) {                                                   // item words are id words
      if (lane == 0) { s_pool_bits[w] = c1; s_pcb_bits[w] = c2; }
    } else {
      if ((c1 >> lane) & 1u) pick_pool(i);
      if ((c2 >> lane) & 1u) pick_pcb(i);
    }
  };
  int32_t *g_m1 = a.ws.unc_id + (int64_t)b * 3 * a.ws.unc_x;       // lists beyond kListCap
  int32_t *g_m2 = g_m1 + a.ws.unc_x;
  classify_words(n, val, sel_pool, w1_lo, w1_hi, sel_pcb, w2_lo, w2_hi, cert, NearLists{s_m1, s_m2, g_m1, g_m2},
                 s_wc, s_tot);
  const int m1c = s_tot[0], m2c = s_tot[1], cert1 = s_tot[2], cert2 = s_tot[3];
  const int32_t *m1 = m1c <= kListCap ? s_m1 : g_m1;
  const int32_t *m2 = m2c <= kListCap ? s_m2 : g_m2;

  // ---- pool.  With two CTAs per sequence (gridDim.y == 2) CTA 0 selects and writes the pool
  // while CTA 1 selects the top-k positions; CTA 1 needs the pool itself only when the
  // candidate blocks outnumber it.
  const bool split = gridDim.y > 1;
  auto run_pool = [&]() {
    if (sel_pool) {
      const bool big = m1c > kListCap;
      int32_t *band = big ? g_m1 + 2 * a.ws.unc_x : s_band;
      float2 *ex = big ? a.ws.unc_val + (int64_t)b * a.ws.unc_x : s_ex;
      auto exact_band = [&](const int32_t *bd, float2 *xv, int u) {
        QFrag f;
        QExact q;
        load_qfrag(qb, wb, lane, f);
        load_qexact(qb, wb, lane, q);
        exact_block_maxima<BLOCK>(a, e, f, q, E, bd, xv, u, id, s_lut);
      };
      resolve_list(m1, m1c, k1, cert1, w1_lo, w1_hi, E, val, id, exact_band, pick_pool, band, ex, s_hist, s_cnt,
                   s_scan, s_out);
    }
    __syncthreads();
    if (sel_pool && !use_bits) {
      cta_sort_asc(s_sort, k1);                                   // k1 <= n_keep <= 4096 ids
      __syncthreads();
    }
  };
  bool pool_done = false;
  if (!split || blockIdx.y == 0) {
    run_pool();
    pool_done = true;
    if (!sel_pool) {
      for (int i = tid; i < n_keep; i += blockDim.x) pool[i] = i < nb ? i : -1;
    } else if (use_bits) {
      emit_bits_ascending(s_pool_bits, nwords, [](int i) { return (int32_t)i; }, pool, n_keep, s_scan);
    } else {
      for (int i = tid; i < n_keep; i += blockDim.x) pool[i] = i < k1 ? s_sort[i] : -1;
    }
    __syncthreads();
    if (split) return;
  }
  // ---- position-candidate blocks: the topk-th largest approximate maximum, lower cut
  if (sel_pcb) {
    const uint32_t kth = list_kth(m2, m2c, [&](int i) { return __float_as_uint(val(i)); }, k2 - cert2,
                                  __float_as_uint(w2_lo), __float_as_uint(w2_hi) - __float_as_uint(w2_lo), s_hist,
                                  s_scan, s_out);
    const float lo2 = lo_cut(__uint_as_float(kth), E);
    for (int j = tid; j < m2c; j += blockDim.x) {
      const int i = m2[j];
      if (val(i) >= lo2) pick_pcb(i);
    }
  }
  __syncthreads();

  // ---- the candidate blocks, ascending, into shared memory
  int32_t *s_list = s_m1;                                          // m1 + m2: 2 kListCap >= kMaxSel ids
  int count;
  if (!sel_pcb) {
    for (int i = tid; i < nb; i += blockDim.x) s_list[i] = i;
    count = nb;
  } else {
    int cnt = 0;
    if (use_bits)
      for (int i = tid; i < nwords; i += blockDim.x) cnt += __popc(s_pcb_bits[i]);
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if (lane == 0) atomicAdd(&s_cnt[kCntPcb], cnt);
    __syncthreads();
    const int n_pcb = s_cnt[kCntPcb];
    if (!use_bits || n_pcb > n_keep) {
      // the pool contains every top-k position's block
      if (!pool_done) run_pool();
      if (!sel_pool) for (int i = tid; i < nb; i += blockDim.x) s_list[i] = i;
      else if (use_bits) emit_bits_ascending(s_pool_bits, nwords, [](int i) { return (int32_t)i; }, s_list, n_keep, s_scan);
      else for (int i = tid; i < k1; i += blockDim.x) s_list[i] = s_sort[i];
      count = k1;
    } else {
      emit_bits_ascending(s_pcb_bits, nwords, [](int i) { return (int32_t)i; }, s_list, n_keep, s_scan);
      count = n_pcb;
    }
  }
  __syncthreads();

  // ---- their positions, with the scan's scores: histogram, then the exact top-k
  const int np = count * BLOCK;
  const bool pstaged = np <= kStageItems;
  uint32_t *s_phist = s_pool_bits;                                  // [kHistBins]
  uint32_t *s_ibits = s_pcb_bits;                                   // item bitmap
  for (int i = tid; i < kHistBins; i += blockDim.x) s_phist[i] = 0u;
  __syncthreads();
  const float *sig = a.sigma_out + (int64_t)b * a.sigma_stride;
  auto pos_of = [&](int i) -> int32_t { return s_list[i / BLOCK] * BLOCK + (i % BLOCK); };
  auto pval = [&](int i) -> float {
    const int32_t pos = pos_of(i);
    return pos < e.len ? __ldcg(sig + pos) : -1.f;
  };
  for (int i0 = tid; i0 < np; i0 += 4 * blockDim.x) {
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) { const int i = i0 + j * blockDim.x; v[j] = i < np ? pval(i) : -1.f; }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + j * blockDim.x;
      if (pstaged && i < np) s_val[i] = v[j];
      if (v[j] >= 0.f) atomicAdd(&s_phist[min(__float_as_uint(v[j]) >> kHistShift, (uint32_t)kHistBins - 1)], 1u);
    }
  }
  __syncthreads();
  cta_find_bins(a.topk, 0, [&](int bin) { return s_phist[bin]; }, s_scan, s_out);
  auto pv = [&](int i) -> float { return pstaged ? s_val[i] : pval(i); };
  const PosWork w{s_hist, s_ibits, s_band, s_band2, s_ex, s_lut, s_cnt, s_scan, s_out, s_wc, s_tot};
  select_positions_core<BLOCK>(a, e, b, np, s_out[4], (uint32_t)s_out[0], pv, pos_of, E, w,
                               a.topk_out + (int64_t)b * a.topk);
}

// Scores of the positions of a block list (the Full layer's candidate blocks, or the pool
// for a Reindex layer), many CTAs per sequence, with their histogram.
template <int BLOCK>
__global__ void __launch_bounds__(256) score_positions_kernel(const __grid_constant__ IdxArgs a) {
  pdl_enter();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const SelUnit u = sel_unit<BLOCK>(a, blockIdx.y);
  const int r = u.r;
  const int32_t *list;
  int count;
  if (a.use_pool) { list = a.pool_in + (int64_t)u.b * a.n_keep; count = a.n_keep; }
  else { list = a.ws.pcb + (int64_t)r * a.n_keep; count = (int)a.ws.pcb_cnt[r]; }
  const int n = count * BLOCK;
  float *pv = a.ws.pvals + (int64_t)r * a.ws.pv_stride;
  QFrag f;
  load_qfrag(a.q + (int64_t)r * kHIdx * kDIdx, a.w + (int64_t)r * kHIdx, lane, f);
  float smx = 0.f;
  score_units<BLOCK>(a, u.e, u.nb_seq, list, n, pv, a.ws.hist2 + (int64_t)r * kHistBins, f, blockIdx.x * 8 + warp,
                     gridDim.x * 8, smx);
  smx = warp_max(smx);
  if (lane == 0 && smx > 0.f) atomicMax(&a.ws.smax2[r], __float_as_uint(smx));
}

// Exact top-k over the scored positions (the Full layer's candidates, or a Reindex pool),
// written ascending.  STAGED: the scores fit in shared memory (n_keep * BLOCK <= kStageItems).
template <int BLOCK, bool STAGED>
__global__ void __launch_bounds__(kSelCta, 1) select_positions_kernel(const __grid_constant__ IdxArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) uint8_t s_dyn[];
  uint32_t *s_hist = reinterpret_cast<uint32_t *>(s_dyn);            // radix scratch [2048]
  uint32_t *s_bits = s_hist + 2048;
  int32_t *s_m = reinterpret_cast<int32_t *>(s_bits + kItemWords);
  int32_t *s_band = s_m + kListCap;
  float2 *s_ex = reinterpret_cast<float2 *>(s_band + kListCap);
  int32_t *s_lut = reinterpret_cast<int32_t *>(s_ex + kListCap);
  int32_t *s_list = s_lut + 256;                                     // [kMaxSel]
  float *s_pv = reinterpret_cast<float *>(s_list + kMaxSel);         // [kStageItems] when STAGED
  __shared__ int s_cnt[8];
  __shared__ int s_scan[72];
  __shared__ int s_out[8];
  __shared__ int s_wc[kSelWarps][4];
  __shared__ int s_tot[4];
  __shared__ float s_E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const SelUnit u = sel_unit<BLOCK>(a, blockIdx.x);
  const int b = u.r;                                                 // q, w, workspace and output slot
  const SeqTable e = u.e;
  const int32_t *list_g;
  int count;
  if (a.use_pool) { list_g = a.pool_in + (int64_t)u.b * a.n_keep; count = a.n_keep; }
  else { list_g = a.ws.pcb + (int64_t)b * a.n_keep; count = (int)a.ws.pcb_cnt[b]; }
  const int n = count * BLOCK;
  const float *pv_g = a.ws.pvals + (int64_t)b * a.ws.pv_stride;     // 16-byte aligned rows
  const uint16_t *qb = a.q + (int64_t)b * kHIdx * kDIdx;
  const float *wb = a.w + (int64_t)b * kHIdx;
  const uint32_t *hist_g = a.ws.hist2 + (int64_t)b * kHistBins;

  if (tid < 8) s_cnt[tid] = 0;
  for (int i = tid; i < count; i += blockDim.x) s_list[i] = __ldg(list_g + i);
  fill_e4m3_lut(s_lut);
  if (warp == 0) {
    const float E = seq_bound(qb, wb, __uint_as_float(a.ws.smax2[b]), lane);
    if (lane == 0) s_E = E;
  }
  if (STAGED) {
    const int n4 = n >> 2;
    for (int i = tid; i < n4; i += blockDim.x)
      reinterpret_cast<float4 *>(s_pv)[i] = __ldcg(reinterpret_cast<const float4 *>(pv_g) + i);
    for (int i = 4 * n4 + tid; i < n; i += blockDim.x) s_pv[i] = __ldcg(pv_g + i);
  }
  // the bin of the topk-th largest score, and the number of valid scores (syncs the staging)
  cta_find_bins(a.topk, 0, [&](int bin) { return __ldcg(hist_g + bin); }, s_scan, s_out);
  const int n_valid = s_out[4];
  const float E = s_E;
  if (a.use_pool)                                                   // the pool must ascend
    for (int i = tid + 1; i < count; i += blockDim.x)
      if (s_list[i] >= 0 && s_list[i - 1] >= s_list[i]) set_err(a.d_err, CSA2_DEVERR_POOL);
  auto val = [&](int i) -> float { return STAGED ? s_pv[i] : __ldcg(pv_g + i); };
  auto pos_of = [&](int i) -> int32_t { return s_list[i / BLOCK] * BLOCK + (i % BLOCK); };
  const PosWork w{s_hist, s_bits, s_m, s_band, s_ex, s_lut, s_cnt, s_scan, s_out, s_wc, s_tot};
  select_positions_core<BLOCK>(a, e, b, n, n_valid, (uint32_t)s_out[0], val, pos_of, E, w,
                               a.topk_out + (int64_t)b * a.topk);
}

// ------------------------------------------------------------------ test: bounds

__global__ void bound_kernel(const __grid_constant__ IdxArgs a, double *bound) {
  const int b = blockIdx.x;
  const float E = seq_bound(a.q + (int64_t)b * kHIdx * kDIdx, a.w + (int64_t)b * kHIdx,
                            __uint_as_float(a.ws.smax[b]), threadIdx.x);
  if (threadIdx.x == 0) bound[b] = (double)E;
  if (b == 0 && threadIdx.x == 0) bound[a.c.B] = (double)kRelF;
}

// ------------------------------------------------------------------ host side

static size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

static int64_t round4(int64_t x) { return (x + 3) & ~(int64_t)3; }

size_t indexer_ws_bytes(int32_t B, int64_t max_len, int32_t block, int32_t n_keep) {
  const int64_t nbm = round4((max_len + block - 1) / block);
  const int64_t npos = round4((int64_t)n_keep * block);
  const int64_t unc = nbm > npos ? nbm : npos;
  size_t z = 2 * align_up((size_t)B * kHistBins * 4) + 4 * align_up((size_t)B * 4);
  size_t s = z;
  s += align_up((size_t)B * nbm * 4);       // bmax
  s += align_up((size_t)B * nbm * 8);       // cand
  s += align_up((size_t)B * n_keep * 4);    // pcb
  s += align_up((size_t)B * npos * 4);      // pvals
  s += align_up((size_t)B * nbm * block * 4);   // sigma
  s += align_up((size_t)B * unc * 12);      // unc_id: three lists per sequence
  s += align_up((size_t)B * unc * 8);       // unc_val
  return s;
}

IndexerWs indexer_ws_carve(void *ws, int32_t B, int64_t max_len, int32_t block, int32_t n_keep) {
  IndexerWs w;
  const int64_t nbm = round4((max_len + block - 1) / block);
  const int64_t npos = round4((int64_t)n_keep * block);
  w.nbm = nbm;
  w.pv_stride = npos;
  w.unc_x = nbm > npos ? nbm : npos;
  char *p = (char *)ws;
  w.hist = (uint32_t *)p; p += align_up((size_t)B * kHistBins * 4);
  w.hist2 = (uint32_t *)p; p += align_up((size_t)B * kHistBins * 4);
  w.smax = (uint32_t *)p; p += align_up((size_t)B * 4);
  w.smax2 = (uint32_t *)p; p += align_up((size_t)B * 4);
  w.cand_cnt = (uint32_t *)p; p += align_up((size_t)B * 4);
  w.pcb_cnt = (uint32_t *)p; p += align_up((size_t)B * 4);
  w.zero_bytes = (size_t)(p - (char *)ws);
  w.bmax = (float *)p; p += align_up((size_t)B * nbm * 4);
  w.cand = (uint64_t *)p; p += align_up((size_t)B * nbm * 8);
  w.pcb = (int32_t *)p; p += align_up((size_t)B * n_keep * 4);
  w.pvals = (float *)p; p += align_up((size_t)B * npos * 4);
  w.sigma = (float *)p; p += align_up((size_t)B * nbm * block * 4);
  w.sigma_stride = nbm * block;
  w.unc_id = (int32_t *)p; p += align_up((size_t)B * w.unc_x * 12);
  w.unc_val = (float2 *)p;
  return w;
}

static size_t scan_smem_bytes(int B, bool priv) {
  return kScanSmem + (priv ? (size_t)kHistBins * 4 : 0) + (size_t)(2 * B + 1) * 8 + (size_t)B * 4;
}

// Long sequences spread their block maxima over few histogram bins, so that global
// atomics on the same addresses serialise; there each CTA counts its home sequence in
// shared memory and adds the counts once at the end.
static bool scan_private_hist(int64_t max_len) { return max_len >= 262144; }

// persistent scan grid: every resident CTA slot of the GPU, capped by the work
template <int BLOCK, bool PRIV>
static int scan_grid_size(int B, int64_t max_len) {
  opt_in_smem((const void *)scan_kernel<BLOCK, false, PRIV>, scan_smem_bytes(CSA2_MAX_B, PRIV), kSiteScanOptin,
              BLOCK * 4 + PRIV * 2 + 0);
  opt_in_smem((const void *)scan_kernel<BLOCK, true, PRIV>, scan_smem_bytes(CSA2_MAX_B, PRIV), kSiteScanOptin,
              BLOCK * 4 + PRIV * 2 + 1);
  const int per_sm = device_memo(kSiteScanOccupancy, ((int64_t)B << 8) | (BLOCK << 1) | (PRIV ? 1 : 0), [B] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scan_kernel<BLOCK, false, PRIV>, kScanWarps * 32,
                                                      scan_smem_bytes(B, PRIV)) != cudaSuccess || n < 1)
      return 1;
    return n;
  });
  const int64_t stages_ub = (int64_t)B * ((max_len + 31) / 32);
  const int64_t g = std::min<int64_t>((stages_ub + kScanWarps - 1) / kScanWarps, (int64_t)num_sms() * per_sm);
  return (int)std::max<int64_t>(g, 1);
}

template <int BLOCK, bool SIGMA>
static void launch_scan(IdxArgs &a, int64_t max_len, cudaStream_t st) {
  const int B = a.c.B;
  if (scan_private_hist(max_len))
    launch_k(scan_kernel<BLOCK, SIGMA, true>, dim3(scan_grid_size<BLOCK, true>(B, max_len)), dim3(kScanWarps * 32),
             scan_smem_bytes(B, true), st, 0, a);
  else
    launch_k(scan_kernel<BLOCK, SIGMA, false>, dim3(scan_grid_size<BLOCK, false>(B, max_len)),
             dim3(kScanWarps * 32), scan_smem_bytes(B, false), st, 0, a);
}

constexpr size_t kFinalizeSmemDirect =
    (size_t)(2048 + 2 * kIdWords) * 4 + (size_t)4 * kListCap * 4 + (size_t)kListCap * 8 + 256 * 4 +
    (size_t)kStageItems * 4;
constexpr size_t kFinalizeSmemCand = kFinalizeSmemDirect + (size_t)kStageItems * 4;
constexpr size_t kSelectSmemBase = (size_t)(2048 + kItemWords) * 4 + (size_t)2 * kListCap * 4 +
                                   (size_t)kListCap * 8 + 256 * 4 + (size_t)kMaxSel * 4;
constexpr size_t kSelectSmemStaged = kSelectSmemBase + (size_t)kStageItems * 4;

template <int BLOCK>
static void select_smem_optin() {
  opt_in_smem((const void *)finalize_blocks_kernel<BLOCK, true>, kFinalizeSmemDirect, kSiteSelectOptin, BLOCK * 4 + 0);
  opt_in_smem((const void *)finalize_blocks_kernel<BLOCK, false>, kFinalizeSmemCand, kSiteSelectOptin, BLOCK * 4 + 1);
  opt_in_smem((const void *)select_positions_kernel<BLOCK, true>, kSelectSmemStaged, kSiteSelectOptin, BLOCK * 4 + 2);
  opt_in_smem((const void *)select_positions_kernel<BLOCK, false>, kSelectSmemBase, kSiteSelectOptin, BLOCK * 4 + 3);
}

// CTAs per row of the position scoring: enough resident warps on every SM, at most 32 per row.
template <int BLOCK>
static int positions_grid(int rows) {
  const int resident = device_memo(kSitePositionsResident, BLOCK, [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, score_positions_kernel<BLOCK>, 256, 0) != cudaSuccess || n < 1)
      n = 2;
    return std::min(n, 4);
  });
  return std::max(1, std::min(32, (int)((int64_t)num_sms() * resident / std::max(rows, 1))));
}

template <int BLOCK>
static void launch_positions(IdxArgs &a, cudaStream_t st) {
  const int B = a.c.B;
  launch_k(score_positions_kernel<BLOCK>, dim3(positions_grid<BLOCK>(B), B), dim3(256), 0, st, 0, a);
  if ((int64_t)a.n_keep * BLOCK <= kStageItems)
    launch_k(select_positions_kernel<BLOCK, true>, dim3(B), dim3(kSelCta), kSelectSmemStaged, st, 0, a);
  else
    launch_k(select_positions_kernel<BLOCK, false>, dim3(B), dim3(kSelCta), kSelectSmemBase, st, 0, a);
}

template <int BLOCK>
static void launch_finalize(IdxArgs &a, cudaStream_t st) {
  const int B = a.c.B;
  const int64_t nbm = a.ws.nbm;
  // pool and top-k positions in separate CTAs while both fit in one wave (one CTA per SM)
  const dim3 fin((unsigned)B, 2 * B <= num_sms() ? 2u : 1u);
  if (nbm <= kDirectBlocks) {
    launch_k(finalize_blocks_kernel<BLOCK, true>, fin, dim3(kSelCta), kFinalizeSmemDirect, st, 0, a);
  } else {
    dim3 cg((unsigned)((nbm + kCollectPer - 1) / kCollectPer), (unsigned)B);
    launch_k(collect_kernel<BLOCK>, cg, dim3(256), 0, st, 0, a);
    launch_k(finalize_blocks_kernel<BLOCK, false>, fin, dim3(kSelCta), kFinalizeSmemCand, st, 0, a);
  }
}

template <int BLOCK>
static cudaError_t full_select_impl(IdxArgs &a, int64_t max_len, const csa2_profile *prof, cudaStream_t st) {
  select_smem_optin<BLOCK>();
  // inside stream capture a timing event must be an external record node
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (prof) cudaStreamIsCapturing(st, &cap);
  const unsigned ev_flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  if (prof) cudaEventRecordWithFlags((cudaEvent_t)prof->start, st, ev_flags);
  launch_scan<BLOCK, true>(a, max_len, st);
  if (prof) cudaEventRecordWithFlags((cudaEvent_t)prof->stop, st, ev_flags);
  launch_finalize<BLOCK>(a, st);
  return cudaGetLastError();
}

// One group of chunked-query rows: rows in uniform groups of 16 are scored on the tensor
// cores, the others by the one-query scan (which sees them through len_scan), then the
// usual finalize on the true row view.
template <int BLOCK>
static cudaError_t chunked_group_impl(IdxArgs &a, const int32_t *len_scan, const CqArgs &cq, int64_t max_len,
                                      cudaStream_t st) {
  select_smem_optin<BLOCK>();
  cudaError_t e = launch_chunk_scores_tc(cq, BLOCK, st);
  if (e != cudaSuccess) return e;
  IdxArgs as = a;
  as.c.seq_len = len_scan;
  launch_scan<BLOCK, true>(as, max_len, st);
  launch_finalize<BLOCK>(a, st);
  return cudaGetLastError();
}

template <int BLOCK>
static cudaError_t verify_impl(IdxArgs &a, int rows, cudaStream_t st) {
  select_smem_optin<BLOCK>();
  launch_k(score_positions_kernel<BLOCK>, dim3(positions_grid<BLOCK>(rows), rows), dim3(256), 0, st, 0, a);
  if ((int64_t)a.n_keep * BLOCK <= kStageItems)
    launch_k(select_positions_kernel<BLOCK, true>, dim3(rows), dim3(kSelCta), kSelectSmemStaged, st, 0, a);
  else
    launch_k(select_positions_kernel<BLOCK, false>, dim3(rows), dim3(kSelCta), kSelectSmemBase, st, 0, a);
  return cudaGetLastError();
}

template <int BLOCK>
static cudaError_t reindex_impl(IdxArgs &a, cudaStream_t st) {
  select_smem_optin<BLOCK>();
  launch_positions<BLOCK>(a, st);
  return cudaGetLastError();
}

// Clears the per-call counters of the workspace (a kernel, so that launches stay chained).
__global__ void zero_ws_kernel(uint4 *p, int64_t n16) {
  pdl_enter();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = make_uint4(0, 0, 0, 0);
}

static cudaError_t zero_ws(const IndexerWs &ws, cudaStream_t st) {
  const int64_t n16 = (int64_t)(ws.zero_bytes / 16);              // zero_bytes is a multiple of 256
  const int64_t grid = std::min<int64_t>((n16 + 1023) / 1024, (int64_t)num_sms() * 4);
  return launch_k(zero_ws_kernel, dim3((unsigned)std::max<int64_t>(grid, 1)), dim3(256), 0, st, 0,
                  reinterpret_cast<uint4 *>(ws.hist), n16);
}

static IdxArgs make_args(const csa2_cache &c, const uint16_t *q, const float *w, int64_t max_len, int n_keep,
                         int topk, const IndexerWs &ws, int32_t *d_err) {
  IdxArgs a;
  a.c = c; a.q = q; a.w = w; a.max_len = max_len; a.n_keep = n_keep; a.topk = topk; a.ws = ws;
  a.pool_out = nullptr; a.pool_in = nullptr; a.topk_out = nullptr;
  a.sigma_out = ws.sigma; a.sigma_stride = ws.sigma_stride;
  a.row_seq = nullptr; a.row_pos = nullptr;
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
  cudaError_t e = zero_ws(ws, st);
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
  cudaError_t e = zero_ws(ws, st);
  if (e != cudaSuccess) return e;
  IdxArgs a = make_args(c, q, w, max_len, n_keep, topk, ws, d_err);
  a.pool_in = pool;
  a.topk_out = topk_idx;
  a.use_pool = 1;
  CSA2_DISPATCH_BLOCK(block, reindex_impl<BL>(a, st));
}

// Verify rows: the Reindex stage per query row (session q_seq[r], causal limit q_pos[r]).
cudaError_t launch_verify_select(const csa2_cache &c, const uint16_t *q, const float *w, const int32_t *q_seq,
                                 const int64_t *q_pos, int64_t T, const int32_t *pool, int block, int n_keep, int topk,
                                 int64_t max_len, int32_t *topk_idx, const IndexerWs &ws, int32_t *d_err,
                                 cudaStream_t st) {
  cudaError_t e = zero_ws(ws, st);
  if (e != cudaSuccess) return e;
  IdxArgs a = make_args(c, q, w, max_len, n_keep, topk, ws, d_err);
  a.pool_in = pool;
  a.topk_out = topk_idx;
  a.use_pool = 1;
  a.row_seq = q_seq;
  a.row_pos = q_pos;
  CSA2_DISPATCH_BLOCK(block, verify_impl<BL>(a, (int)T, st));
}

// Chunked queries: every query row gets the Full selection over its session's positions up
// to its own.  A small kernel turns (session, position) into a per-row view of the cache
// (the session's base, length position + 1) and marks the rows whose group of 16 shares one
// session: those are scored on the tensor cores, the rest by the one-query scan (which sees
// them through len_scan).  Groups of up to CSA2_MAX_B rows then run the selection on that
// view, the rows of a group sharing one workspace.
__global__ void row_tables_kernel(const csa2_cache c, const int32_t *q_seq, const int64_t *q_pos, int64_t T,
                                  int64_t max_len, int64_t *base_v, int32_t *len_v, int32_t *len_scan,
                                  int32_t *d_err) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;            // a multiple of 32
  for (int64_t r0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); r0 < T; r0 += stride) {
    const int64_t r = r0 + lane;
    int64_t base = 0;
    int32_t len = 0;
    if (r < T) {
      const int b = q_seq[r];
      const int64_t p = q_pos[r];
      if (b < 0 || b >= c.B) {
        set_err(d_err, CSA2_DEVERR_SEQ);
      } else if (p < 0 || p >= (int64_t)c.seq_len[b]) {
        set_err(d_err, CSA2_DEVERR_POS);
      } else if (p + 1 > max_len || c.seq_base[b] < 0 || c.seq_base[b] + c.seq_len[b] > c.T_cap) {
        set_err(d_err, CSA2_DEVERR_LEN);                            // the row reads nothing
      } else {
        base = c.seq_base[b];
        len = (int32_t)(p + 1);
      }
      base_v[r] = base;
      len_v[r] = len;
    }
    // r0 is a multiple of 32: lanes 0-15 and 16-31 each hold one group of 16 rows
    const int64_t b0 = __shfl_sync(0xffffffffu, base, lane & 16);
    const unsigned same = __ballot_sync(0xffffffffu, r >= T || base == b0);
    const bool uniform = ((same >> (lane & 16)) & 0xFFFFu) == 0xFFFFu;
    if (r < T) len_scan[r] = uniform ? 0 : len;
  }
}

constexpr int64_t kChunkRows = CSA2_MAX_B;

size_t chunked_ws_bytes(int64_t T, int64_t max_len, int32_t block, int32_t n_keep) {
  const int32_t G = (int32_t)std::min<int64_t>(std::max<int64_t>(T, 1), kChunkRows);
  return align_up((size_t)T * 8) + 2 * align_up((size_t)T * 4) + indexer_ws_bytes(G, max_len, block, n_keep);
}

cudaError_t launch_chunked_select(const csa2_cache &c, const uint16_t *q, const float *w, const int32_t *q_seq,
                                  const int64_t *q_pos, int64_t T, int block, int n_keep, int topk, int64_t max_len,
                                  int32_t *pool, int32_t *topk_idx, void *ws, int32_t *d_err, cudaStream_t st) {
  int64_t *base_v = reinterpret_cast<int64_t *>(ws);
  int32_t *len_v = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(ws) + align_up((size_t)T * 8));
  int32_t *len_scan = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(len_v) + align_up((size_t)T * 4));
  void *iws = reinterpret_cast<char *>(len_scan) + align_up((size_t)T * 4);
  const int32_t G = (int32_t)std::min<int64_t>(T, kChunkRows);
  const IndexerWs iw = indexer_ws_carve(iws, G, max_len, block, n_keep);
  const unsigned grid = (unsigned)std::min<int64_t>((T + 255) / 256, (int64_t)num_sms() * 4);
  cudaError_t e = launch_k(row_tables_kernel, dim3(grid), dim3(256), 0, st, 0, c, q_seq, q_pos, T, max_len, base_v,
                           len_v, len_scan, d_err);
  for (int64_t g0 = 0; e == cudaSuccess && g0 < T; g0 += kChunkRows) {
    csa2_cache cg = c;
    cg.B = (int32_t)std::min<int64_t>(kChunkRows, T - g0);
    cg.seq_base = base_v + g0;
    cg.seq_len = len_v + g0;
    e = zero_ws(iw, st);
    if (e != cudaSuccess) break;
    IdxArgs a = make_args(cg, q + g0 * kHIdx * kDIdx, w + g0 * kHIdx, max_len, n_keep, topk, iw, d_err);
    a.pool_out = pool + g0 * n_keep;
    a.pool_in = a.pool_out;
    a.topk_out = topk_idx + g0 * topk;
    CqArgs cq;
    cq.ik_codes = c.ik_codes; cq.ik_scale = c.ik_scale;
    cq.base_v = base_v + g0; cq.len_v = len_v + g0;
    cq.q = a.q; cq.w = a.w; cq.n = cg.B; cq.ws = iw; cq.d_err = d_err;
    const int32_t *ls = len_scan + g0;
    auto run = [&]() -> cudaError_t { CSA2_DISPATCH_BLOCK(block, chunked_group_impl<BL>(a, ls, cq, max_len, st)); };
    e = run();
  }
  return e;
}

// Test: the tensor-core scores of up to CSA2_MAX_B chunked-query rows (each row's group of
// 16 must share a session) into sigma [T][max_len], with the per-row bound as for the scan.
cudaError_t launch_test_chunk_scores(const csa2_cache &c, const uint16_t *q, const float *w, const int32_t *q_seq,
                                     const int64_t *q_pos, int64_t T, int64_t max_len, float *sigma, double *bound,
                                     void *ws, int32_t *d_err, cudaStream_t st) {
  int64_t *base_v = reinterpret_cast<int64_t *>(ws);
  int32_t *len_v = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(ws) + align_up((size_t)T * 8));
  int32_t *len_scan = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(len_v) + align_up((size_t)T * 4));
  void *iws = reinterpret_cast<char *>(len_scan) + align_up((size_t)T * 4);
  IndexerWs iw = indexer_ws_carve(iws, (int32_t)T, max_len, 8, 1);
  cudaError_t e = launch_k(row_tables_kernel, dim3(1), dim3(1024), 0, st, 0, c, q_seq, q_pos, T, max_len, base_v,
                           len_v, len_scan, d_err);
  if (e == cudaSuccess) e = zero_ws(iw, st);
  if (e != cudaSuccess) return e;
  iw.sigma = sigma;
  iw.sigma_stride = max_len;
  CqArgs cq;
  cq.ik_codes = c.ik_codes; cq.ik_scale = c.ik_scale;
  cq.base_v = base_v; cq.len_v = len_v; cq.q = q; cq.w = w; cq.n = (int)T; cq.ws = iw; cq.d_err = d_err;
  e = launch_chunk_scores_tc(cq, 8, st);
  if (e != cudaSuccess) return e;
  csa2_cache cv = c;
  cv.B = (int32_t)T;
  cv.seq_base = base_v;
  cv.seq_len = len_v;
  IdxArgs a = make_args(cv, q, w, max_len, 1, 1, iw, d_err);
  bound_kernel<<<(unsigned)T, 32, 0, st>>>(a, bound);
  return cudaGetLastError();
}

cudaError_t launch_test_scores(const csa2_cache &c, const uint16_t *q, const float *w, int64_t max_len,
                               float *sigma, double *bound, const IndexerWs &ws, int32_t *d_err,
                               cudaStream_t st) {
  cudaError_t e = zero_ws(ws, st);
  if (e != cudaSuccess) return e;
  IdxArgs a = make_args(c, q, w, max_len, 1, 1, ws, d_err);
  a.sigma_out = sigma;
  a.sigma_stride = max_len;
  const int B = c.B;
  launch_scan<8, true>(a, max_len, st);
  bound_kernel<<<B, 32, 0, st>>>(a, bound);
  return cudaGetLastError();
}

}  // namespace csa2
