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
constexpr int kMaxSel = 4096;                          // n_keep_blocks limit

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
  float *sigma_out;         // test: [B][max_len]
  int32_t *d_err;
  int32_t use_pool;         // position stage reads pool_in instead of the candidate list
};

// ------------------------------------------------------------------ scan

// Each warp streams a contiguous range of 16-position units through its own cp.async
// ring in shared memory (kScanStages stages of 32 rows), so loads in flight hold no
// registers.  A warp's range is walked as per-sequence segments; a stage never mixes
// sequences.  Stage layout: 32 rows x 64 key bytes, then 32 scales stored so that lane
// quad g finds rows g, g+8, g+16, g+24 in one 16-byte word.
#ifndef CSA2_SCAN_WARPS
#define CSA2_SCAN_WARPS 8
#endif
#ifndef CSA2_SCAN_STAGES
#define CSA2_SCAN_STAGES 4
#endif
#ifndef CSA2_SCAN_CTAS
#define CSA2_SCAN_CTAS 3
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
// one redux over the lanes of each block, then the block's first lane writes it.
template <int BLOCK>
__device__ __forceinline__ void emit_stage(float o, int lane, int64_t cp, int rows, int64_t L, float *bmax,
                                           uint32_t *hist) {
  const int g = lane >> 2, t = lane & 3;
  unsigned mask;
  if constexpr (BLOCK == 16) mask = t < 2 ? 0x33333333u : 0xCCCCCCCCu;
  else mask = (0x11111111u >> (32 - 4 * BLOCK)) << (t + 4 * BLOCK * (g / BLOCK));
  const uint32_t m = __reduce_max_sync(mask, __float_as_uint(o));       // scores are >= 0: bit order = value order
  const int row = 8 * t + g;
  const bool writer = BLOCK == 16 ? (g == 0 && (t & 1) == 0) : (g % BLOCK) == 0;
  if (writer && row < rows && cp + row < L) {
    bmax[(cp + row) / BLOCK] = __uint_as_float(m);
    atomicAdd(&hist[min(m >> kHistShift, (uint32_t)kHistBins - 1)], 1u);
  }
}

template <int BLOCK>
__global__ void __launch_bounds__(kScanWarps * 32, CSA2_SCAN_CTAS) scan_kernel(const __grid_constant__ IdxArgs a) {
  extern __shared__ __align__(16) uint8_t s_dyn[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = a.c.B;
  int64_t *s_units = reinterpret_cast<int64_t *>(s_dyn + kScanSmem);
  int64_t *s_base = s_units + (B + 1);
  int32_t *s_len = reinterpret_cast<int32_t *>(s_base + B);
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
  const int64_t per = (total + W - 1) / W;
  const int64_t u_begin = min(total, gw * per), u_end = min(total, u_begin + per);
  if (u_begin >= u_end) return;
  const int g = lane >> 2, t = lane & 3;
  const uint8_t *ik_codes = a.c.ik_codes;
  const float *ik_scale = a.c.ik_scale;

  int b0;
  {
    int lo = 0, hi = B;                                          // s_units[lo] <= u_begin < s_units[hi]
    while (hi - lo > 1) { int mid = (lo + hi) >> 1; if (s_units[mid] <= u_begin) lo = mid; else hi = mid; }
    b0 = lo;
  }
  // producer cursor: sequence, next position, units left in this segment / in the warp
  int pb = b0;
  int64_t pp = (u_begin - s_units[b0]) * 16;
  int64_t pleft = u_end - u_begin;
  int64_t pseg = min(pleft, s_units[b0 + 1] - u_begin);
  uint8_t *ring = s_dyn + warp * kScanSmemPerWarp;
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
  uint32_t issued = 0;

  auto issue_stage = [&]() {
    const uint32_t dst = ring_s + (issued % kScanStages) * kStageBytes;
    ++issued;
    int k = 0;
    if (pleft > 0) {
      if (pseg == 0) {                                           // next sequence with work
        do { ++pb; } while (s_units[pb + 1] == s_units[pb]);
        pp = 0;
        pseg = min(pleft, s_units[pb + 1] - s_units[pb]);
      }
      k = (int)min((int64_t)2, pseg);
    }
    const int64_t L = k ? s_len[pb] : 0;
    const int64_t base = k ? s_base[pb] : 0;
    const int lim = (int)min((int64_t)(16 * k), L - pp);            // rows of this stage inside the sequence
    const uint8_t *src = ik_codes + (base + pp) * kDIdx + 16 * t;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = g + 8 * q;
      const bool v = r < lim;
      cp_async16(dst + r * kDIdx + 16 * t, v ? src + r * kDIdx : ik_codes, v);
    }
    const bool vs = lane < lim;
    cp_async4(dst + kStageRows * kDIdx + 4 * ((lane & 7) * 4 + (lane >> 3)), vs ? ik_scale + base + pp + lane : ik_scale,
              vs);
    cp_async_commit();
    pp += 16 * k;
    pseg -= k;
    pleft -= k;
  };
#pragma unroll
  for (int s = 0; s < kScanStages - 1; ++s) issue_stage();

  // consumer cursor mirrors the producer
  int cb = b0;
  int64_t cp = (u_begin - s_units[b0]) * 16;
  int64_t cleft = u_end - u_begin;
  int64_t cseg = min(cleft, s_units[b0 + 1] - u_begin);
  uint32_t consumed = 0;
  QFrag f;
  int cur_b = -1;
  float smx = 0.f;
  float *bmax = nullptr;
  uint32_t *hist = nullptr;
  int64_t L = 0;
  while (cleft > 0) {
    issue_stage();
    cp_async_wait<kScanStages - 1>();
    __syncwarp();
    if (cseg == 0) {
      do { ++cb; } while (s_units[cb + 1] == s_units[cb]);
      cp = 0;
      cseg = min(cleft, s_units[cb + 1] - s_units[cb]);
    }
    const int k = (int)min((int64_t)2, cseg);
    const uint8_t *st = ring + (consumed % kScanStages) * kStageBytes;
    ++consumed;
    const uint4 ka = *reinterpret_cast<const uint4 *>(st + g * kDIdx + 16 * t);
    const uint4 ka8 = *reinterpret_cast<const uint4 *>(st + (g + 8) * kDIdx + 16 * t);
    const uint4 kb = *reinterpret_cast<const uint4 *>(st + (g + 16) * kDIdx + 16 * t);
    const uint4 kb8 = *reinterpret_cast<const uint4 *>(st + (g + 24) * kDIdx + 16 * t);
    const float4 sc = *reinterpret_cast<const float4 *>(st + kStageRows * kDIdx + 16 * g);
    __syncwarp();
    if (cb != cur_b) {                                           // a new sequence: its queries and weights
      if (cur_b >= 0) {
        const float m = warp_max(smx);
        if (lane == 0) atomicMax(&a.ws.smax[cur_b], __float_as_uint(m));
      }
      load_qfrag(a.q + (int64_t)cb * kHIdx * kDIdx, a.w + (int64_t)cb * kHIdx, lane, f);
      cur_b = cb;
      smx = 0.f;
      bmax = a.ws.bmax + (int64_t)cb * a.ws.nbm;
      hist = a.ws.hist + (int64_t)cb * kHistBins;
      L = s_len[cb];
    }
    const float o = score32_row(f, ka, ka8, kb, kb8, sc, t);
    smx = fmaxf(smx, fmaxf(fmaxf(sc.x, sc.y), fmaxf(sc.z, sc.w)));
    const int row = 8 * t + g;
    if (a.sigma_out && row < 16 * k && cp + row < L) a.sigma_out[(int64_t)cb * a.max_len + cp + row] = o;
    emit_stage<BLOCK>(o, lane, cp, 16 * k, L, bmax, hist);
    cp += 16 * k;
    cseg -= k;
    cleft -= k;
  }
  cp_async_wait<0>();
  if (cur_b >= 0) {
    const float m = warp_max(smx);
    if (lane == 0) atomicMax(&a.ws.smax[cur_b], __float_as_uint(m));
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
  constexpr int kPer = kCollectPer / 256;
  __shared__ int s_scan[8];
  __shared__ int s_misc[4];
  __shared__ double s_E;
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
      double E = seq_bound(a.q + (int64_t)b * kHIdx * kDIdx, a.w + (int64_t)b * kHIdx,
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

// ------------------------------------------------------------------ block finalisation and positions

constexpr int kSelCta = 256;           // threads of the per-sequence selection kernels
constexpr int kBitmapWords = 4096;     // one bit per block: 131,072 blocks (1M positions at block 8)
constexpr int kCandSmem = 8192;        // candidates staged in shared memory (64 KB)
constexpr int kPvalSmem = 16384;       // position scores staged in shared memory (64 KB)
constexpr int kUncSmem = 1024;         // band entries kept in shared memory (more spill to global)
constexpr int kFlagWords = kMaxSel * 16 / 32;   // one bit per candidate position (<= 65,536)

// Approximate scores of the positions of an ascending block list (units of 16 positions;
// this warp takes units u_first, u_first + u_step, ...; the loads of four units are issued
// before any arithmetic).  Invalid positions score -1.
template <int BLOCK>
__device__ void score_units(const IdxArgs &a, const SeqTable &e, int64_t nb, const int32_t *list, int n, float *pv,
                            const QFrag &f, int u_first, int u_step, float &smx) {
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
      float o0, o1;
      score16(f, k[j][0], k[j][1], s[j][0], s[j][1], o0, o1);
      smx = fmaxf(smx, fmaxf(s[j][0], s[j][1]));
      if (t == 0) {
        const int i0 = (u0 + j * u_step) * 16 + g;
        if (i0 < n) pv[i0] = ok[j][0] ? o0 : -1.f;
        if (i0 + 8 < n) pv[i0 + 8] = ok[j][1] ? o1 : -1.f;
      }
    }
  }
}

// Ranks `u` band entries (ids ascending <=> ties to the lower id) by exact score and calls
// pick(id) for those of rank < need.
template <class PickFn>
__device__ void rank_band(const int32_t *ids, const float2 *vals, int u, int need, PickFn pick) {
  for (int i = threadIdx.x; i < u; i += blockDim.x) {
    const float2 vi = vals[i];
    const int32_t ii = ids[i];
    int rank = 0;
    for (int m = 0; m < u; ++m) {
      const float2 vm = vals[m];
      rank += df_greater(vm, vi) || (df_equal(vm, vi) && ids[m] < ii);
    }
    if (rank < need) pick(ii);
  }
}

// Exact maxima of `u` band blocks, one warp per block.  The block's rows are first scored
// on the tensor cores; only rows whose upper bound reaches the best lower bound of the
// block are rescored exactly (usually one).
template <int BLOCK>
__device__ void exact_block_maxima(const IdxArgs &a, const SeqTable &e, const QFrag &f, const QExact &q, double E,
                                   const int32_t *unc_id, float2 *unc_val, int u, const int32_t *lut) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  for (int i = warp; i < u; i += nwarps) {
    const int32_t j = unc_id[i];
    float best_lo = 0.f;
    float2 best = make_float2(-1.f, 0.f);
    for (int r0 = 0; r0 < BLOCK; r0 += 16) {                 // 16 rows per pass (one for BLOCK <= 8)
      const int rg = r0 + g, rg8 = r0 + g + 8;
      const int64_t p0 = (int64_t)j * BLOCK + rg, p8 = (int64_t)j * BLOCK + rg8;
      const bool v0 = rg < BLOCK && p0 < e.len, v8 = rg8 < BLOCK && p8 < e.len;
      const uint4 k0 = v0 ? ld_nc16(a.c.ik_codes + (e.base + p0) * kDIdx + 16 * t) : make_uint4(0, 0, 0, 0);
      const uint4 k8 = v8 ? ld_nc16(a.c.ik_codes + (e.base + p8) * kDIdx + 16 * t) : make_uint4(0, 0, 0, 0);
      const float s0 = v0 ? __ldg(a.c.ik_scale + e.base + p0) : 0.f;
      const float s8 = v8 ? __ldg(a.c.ik_scale + e.base + p8) : 0.f;
      float o0, o8;
      score16(f, k0, k8, s0, s8, o0, o8);
      // bounds of each row's exact score
      const float lo0 = v0 ? __double2float_rd((1.0 - 2.0 * kRel) * o0 - E) : -FLT_MAX;
      const float lo8 = v8 ? __double2float_rd((1.0 - 2.0 * kRel) * o8 - E) : -FLT_MAX;
      best_lo = fmaxf(best_lo, warp_max(fmaxf(lo0, lo8)));
      const float hi0 = v0 ? __double2float_ru((1.0 + 2.0 * kRel) * o0 + E) : -FLT_MAX;
      const float hi8 = v8 ? __double2float_ru((1.0 + 2.0 * kRel) * o8 + E) : -FLT_MAX;
      // rows that can still be the block's maximum
      unsigned cand = __ballot_sync(0xffffffffu, t == 0 && v0 && hi0 >= best_lo) & 0x11111111u;
      unsigned cand8 = __ballot_sync(0xffffffffu, t == 0 && v8 && hi8 >= best_lo) & 0x11111111u;
      while (cand | cand8) {
        const bool from8 = cand == 0u;
        const int src = __ffs(from8 ? cand8 : cand) - 1;      // lane of the quad holding the row
        if (from8) cand8 &= cand8 - 1; else cand &= cand - 1;
        const uint4 kk = make_uint4(__shfl_sync(0xffffffffu, from8 ? k8.x : k0.x, src + t),
                                    __shfl_sync(0xffffffffu, from8 ? k8.y : k0.y, src + t),
                                    __shfl_sync(0xffffffffu, from8 ? k8.z : k0.z, src + t),
                                    __shfl_sync(0xffffffffu, from8 ? k8.w : k0.w, src + t));
        const float ss = __shfl_sync(0xffffffffu, from8 ? s8 : s0, src);
        const float2 v = exact_sigma(q, kk, ss, lut);
        if (df_greater(v, best)) best = v;
      }
    }
    if (lane == 0) unc_val[i] = best;
  }
}

// Exact top-k positions among n candidates with approximate scores pv[i] (-1 invalid);
// candidate i is position list[i/BLOCK]*BLOCK + i%BLOCK, ascending in i.  Writes the
// selected positions ascending to out[0..topk), -1 padded.  Every thread calls it.
struct SelSmem {
  uint32_t *hist;      // [4096]
  uint32_t *flag;      // [n/32]
  int32_t *unc_id;     // [kUncSmem]
  float2 *unc_val;     // [kUncSmem]
  int *cnt;            // [8]
  int *scan;           // [72]
  int *out;            // [4]
  const int32_t *lut;  // [256]
};

template <int BLOCK>
__device__ void select_topk(const IdxArgs &a, const SeqTable &e, int b, const int32_t *list, int n, const float *pv,
                            double E, int32_t *out, const SelSmem &sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int nwords = (n + 31) / 32;
  auto pos_of = [&](int i) -> int32_t { return list[i / BLOCK] * BLOCK + (i % BLOCK); };
  for (int i = tid; i < nwords; i += blockDim.x) sm.flag[i] = 0u;
  for (int i = tid; i < kHistBins; i += blockDim.x) sm.hist[i] = 0u;
  if (tid < 8) sm.cnt[tid] = 0;
  __syncthreads();
  const int iters = (n + blockDim.x - 1) / blockDim.x;
  int nvalid = 0;
  for (int it = 0; it < iters; ++it) {                       // histogram of the valid scores
    const int i = it * blockDim.x + tid;
    const float v = i < n ? pv[i] : -1.f;
    const bool valid = v >= 0.f;
    const unsigned act = __ballot_sync(0xffffffffu, valid);
    nvalid += __popc(act);
    if (valid) {
      const uint32_t bin = min(score_key(v) >> kHistShift, (uint32_t)kHistBins - 1);
      const unsigned grp = __match_any_sync(act, bin);
      if (lane == __ffs(grp) - 1) atomicAdd(&sm.hist[bin], (uint32_t)__popc(grp));
    }
  }
  if (lane == 0) atomicAdd(&sm.cnt[3], nvalid);
  __syncthreads();
  const int n_valid = sm.cnt[3];
  const int k = min(a.topk, n_valid);
  if (n_valid <= a.topk) {
    for (int i = tid; i < n; i += blockDim.x)
      if (pv[i] >= 0.f) atomicOr(&sm.flag[i >> 5], 1u << (i & 31));
  } else {
    cta_find_bin(kHistBins, k, [&](int bin) { return sm.hist[bin]; }, sm.scan, sm.out);
    const uint32_t bin = (uint32_t)sm.out[0];
    const int above = sm.out[1];
    const uint32_t kth =
        cta_kth_in_bin(n, k - above, [&](int i) { return pv[i] >= 0.f ? score_key(pv[i]) : 0u; }, bin, sm.hist,
                       sm.scan, sm.out);
    const float theta = __uint_as_float(kth);
    const float hi = hi_cut(theta, E), lo = lo_cut(theta, E);
    int32_t *g_id = a.ws.unc_id + (int64_t)b * a.ws.unc_cap;
    float2 *g_val = a.ws.unc_val + (int64_t)b * a.ws.unc_cap;
    for (int it = 0; it < iters; ++it) {
      const int i = it * blockDim.x + tid;
      const float v = i < n ? pv[i] : -1.f;
      const bool in = v >= 0.f && v > hi;
      const bool unc = v >= 0.f && !in && v >= lo;
      if (warp_reserve(in, &sm.cnt[0]) >= 0) atomicOr(&sm.flag[i >> 5], 1u << (i & 31));
      const int su = warp_reserve(unc, &sm.cnt[1]);
      if (unc) {
        if (su < kUncSmem) sm.unc_id[su] = i; else g_id[su] = i;   // candidate index, ascending = position order
      }
    }
    __syncthreads();
    const int n_in = sm.cnt[0], u = sm.cnt[1];
    const bool small = u <= kUncSmem;
    int32_t *ids = small ? sm.unc_id : g_id;
    float2 *vals = small ? sm.unc_val : g_val;
    if (!small)
      for (int i = tid; i < kUncSmem; i += blockDim.x) g_id[i] = sm.unc_id[i];
    __syncthreads();
    if (u > 0) {
      QExact q;
      load_qexact(a.q + (int64_t)b * kHIdx * kDIdx, a.w + (int64_t)b * kHIdx, lane, q);
      for (int i = warp; i < u; i += nwarps) {
        const int64_t row = e.base + pos_of(ids[i]);
        const uint4 kk = __ldg(reinterpret_cast<const uint4 *>(a.c.ik_codes + row * kDIdx + 16 * (lane & 3)));
        const float2 v = exact_sigma(q, kk, __ldg(a.c.ik_scale + row), sm.lut);
        if (lane == 0) vals[i] = v;
      }
    }
    __syncthreads();
    rank_band(ids, vals, u, k - n_in, [&](int32_t ii) { atomicOr(&sm.flag[ii >> 5], 1u << (ii & 31)); });
  }
  __syncthreads();
  emit_bits_ascending(sm.flag, nwords, pos_of, out, a.topk, sm.scan);
}

// The Full layer after the scan: the pool (top n_keep blocks, exact) and the ascending list
// of blocks that may hold a top-k position (every block whose upper bound reaches the
// lower bound of the k-th largest block maximum).
template <int BLOCK>
__global__ void __launch_bounds__(kSelCta) finalize_blocks_kernel(const __grid_constant__ IdxArgs a) {
  extern __shared__ __align__(16) uint64_t s_cand[];
  __shared__ uint32_t s_hist[1024];
  __shared__ uint32_t s_bits[kBitmapWords];
  __shared__ int32_t s_unc_id[kUncSmem];
  __shared__ float2 s_unc_val[kUncSmem];
  __shared__ int32_t s_lut[256];
  __shared__ int s_cnt[8];
  __shared__ int s_scan[72];
  __shared__ int s_out[4];
  __shared__ double s_E;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const SeqTable e = seq_entry(a.c, b, a.max_len, nullptr);
  const int64_t nb = (e.len + BLOCK - 1) / BLOCK;
  const int n_keep = a.n_keep;
  const int k1 = (int)min((int64_t)n_keep, nb);
  const int c = (int)a.ws.cand_cnt[b];
  const uint64_t *cand_g = a.ws.cand + (int64_t)b * a.ws.nbm;
  const uint32_t *hist_g = a.ws.hist + (int64_t)b * kHistBins;
  int32_t *pool = a.pool_out + (int64_t)b * n_keep;
  int32_t *pcb = a.ws.pcb + (int64_t)b * n_keep;
  const uint16_t *qb = a.q + (int64_t)b * kHIdx * kDIdx;
  const float *wb = a.w + (int64_t)b * kHIdx;
  const bool use_bits = nb <= (int64_t)kBitmapWords * 32;
  const int nwords = (int)((nb + 31) / 32);
  const bool staged = c <= kCandSmem;
  if (staged)
    for (int i = tid; i < c; i += blockDim.x) s_cand[i] = __ldcg(cand_g + i);
  const uint64_t *cand = staged ? s_cand : cand_g;
  fill_e4m3_lut(s_lut);
  if (warp == 0) {
    double E = seq_bound(qb, wb, __uint_as_float(a.ws.smax[b]), lane);
    if (lane == 0) s_E = E;
  }
  if (tid < 8) s_cnt[tid] = 0;
  if (use_bits)
    for (int i = tid; i < nwords; i += blockDim.x) s_bits[i] = 0u;
  __syncthreads();
  const double E = s_E;
  const int iters = (c + blockDim.x - 1) / blockDim.x;
  auto cval = [&](int i) { return __uint_as_float((uint32_t)(cand[i] >> 32)); };
  auto ckey = [&](int i) { return (uint32_t)(cand[i] >> 32); };
  auto cid = [&](int i) { return (int32_t)(uint32_t)cand[i]; };
  int32_t *list_fallback = a.ws.unc_id + (int64_t)b * a.ws.unc_cap;   // only without the bitmap
  auto mark = [&](int32_t j, int slot) {
    if (use_bits) atomicOr(&s_bits[j >> 5], 1u << (j & 31));
    else if (slot >= 0) list_fallback[slot] = j;
  };
  // the k-th largest approximate block maximum: its histogram bin, then two radix passes
  auto kth_block = [&](int k) {
    cta_find_bin(kHistBins, k, [&](int bin) { return __ldcg(hist_g + bin); }, s_scan, s_out);
    const uint32_t bin = (uint32_t)s_out[0];
    const int above = s_out[1];
    return __uint_as_float(cta_kth_in_bin(c, k - above, ckey, bin, s_hist, s_scan, s_out));
  };

  // ---- pool: the top k1 blocks by (exact block score desc, id asc)
  if (nb <= n_keep) {
    for (int i = tid; i < n_keep; i += blockDim.x) pool[i] = i < nb ? i : -1;
  } else {
    const float theta = kth_block(k1);
    const float hi = hi_cut(theta, E), lo = lo_cut(theta, E);
    int32_t *g_id = a.ws.unc_id + (int64_t)b * a.ws.unc_cap + a.ws.nbm;       // past the fallback list
    float2 *g_val = a.ws.unc_val + (int64_t)b * a.ws.unc_cap;
    for (int it = 0; it < iters; ++it) {
      const int i = it * blockDim.x + tid;
      const float v = i < c ? cval(i) : -1.f;
      const bool in = i < c && v > hi;
      const bool unc = i < c && !in && v >= lo;
      const int s_in = warp_reserve(in, &s_cnt[0]);
      if (in) mark(cid(i), s_in);
      const int s_un = warp_reserve(unc, &s_cnt[1]);
      if (unc) {
        if (s_un < kUncSmem) s_unc_id[s_un] = cid(i); else g_id[s_un] = cid(i);
      }
    }
    __syncthreads();
    const int n_in = s_cnt[0], u = s_cnt[1];
    const bool small = u <= kUncSmem;
    int32_t *ids = small ? s_unc_id : g_id;
    float2 *vals = small ? s_unc_val : g_val;
    if (!small)
      for (int i = tid; i < kUncSmem; i += blockDim.x) g_id[i] = s_unc_id[i];
    __syncthreads();
    if (u > 0) {
      QFrag f;
      QExact q;
      load_qfrag(qb, wb, lane, f);
      load_qexact(qb, wb, lane, q);
      exact_block_maxima<BLOCK>(a, e, f, q, E, ids, vals, u, s_lut);
    }
    __syncthreads();
    rank_band(ids, vals, u, k1 - n_in, [&](int32_t ji) {
      if (use_bits) atomicOr(&s_bits[ji >> 5], 1u << (ji & 31));
      else list_fallback[atomicAdd(&s_cnt[0], 1)] = ji;
    });
    __syncthreads();
    if (use_bits) {
      emit_bits_ascending(s_bits, nwords, [](int i) { return (int32_t)i; }, pool, n_keep, s_scan);
    } else {
      // without the bitmap (more than 131,072 blocks): order the k1 ids through the global list
      __syncthreads();
      for (int i = tid; i < n_keep; i += blockDim.x) pool[i] = i < k1 ? list_fallback[i] : -1;
      __syncthreads();
      if (tid == 0) {   // insertion sort of at most n_keep ids; this path serves contexts > 1M at block 8
        for (int i = 1; i < k1; ++i) {
          const int32_t v = pool[i];
          int j = i - 1;
          while (j >= 0 && pool[j] > v) { pool[j + 1] = pool[j]; --j; }
          pool[j + 1] = v;
        }
      }
    }
  }
  __syncthreads();

  // ---- position-candidate blocks (ascending)
  if (nb <= a.topk) {
    for (int i = tid; i < n_keep; i += blockDim.x) pcb[i] = i < nb ? i : -1;
    if (tid == 0) a.ws.pcb_cnt[b] = (uint32_t)nb;
    return;
  }
  const float lo2 = lo_cut(kth_block(a.topk), E);
  if (use_bits)
    for (int i = tid; i < nwords; i += blockDim.x) s_bits[i] = 0u;
  if (tid == 0) s_cnt[2] = 0;
  __syncthreads();
  for (int it = 0; it < iters; ++it) {
    const int i = it * blockDim.x + tid;
    const bool keep = i < c && cval(i) >= lo2;
    const int slot = warp_reserve(keep, &s_cnt[2]);
    if (keep) mark(cid(i), slot);
  }
  __syncthreads();
  const int n_pcb = s_cnt[2];
  if (n_pcb > n_keep || !use_bits) {
    // a pathological band (or no bitmap): the pool always contains them, already ascending
    for (int i = tid; i < n_keep; i += blockDim.x) pcb[i] = pool[i];
    if (tid == 0) a.ws.pcb_cnt[b] = (uint32_t)k1;
  } else {
    emit_bits_ascending(s_bits, nwords, [](int i) { return (int32_t)i; }, pcb, n_keep, s_scan);
    if (tid == 0) a.ws.pcb_cnt[b] = (uint32_t)n_pcb;
  }
}

// Scores of the positions of a block list (the Full layer's candidate blocks, or the pool
// for a Reindex layer), many CTAs per sequence.
template <int BLOCK>
__global__ void __launch_bounds__(256) score_positions_kernel(const __grid_constant__ IdxArgs a) {
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const SeqTable e = seq_entry(a.c, b, a.max_len, nullptr);
  const int64_t nb = (e.len + BLOCK - 1) / BLOCK;
  const int32_t *list;
  int count;
  if (a.use_pool) { list = a.pool_in + (int64_t)b * a.n_keep; count = a.n_keep; }
  else { list = a.ws.pcb + (int64_t)b * a.n_keep; count = (int)a.ws.pcb_cnt[b]; }
  const int n = count * BLOCK;
  float *pv = a.ws.pvals + (int64_t)b * a.n_keep * BLOCK;
  QFrag f;
  load_qfrag(a.q + (int64_t)b * kHIdx * kDIdx, a.w + (int64_t)b * kHIdx, lane, f);
  float smx = 0.f;
  score_units<BLOCK>(a, e, nb, list, n, pv, f, blockIdx.x * 8 + warp, gridDim.x * 8, smx);
  smx = warp_max(smx);
  if (lane == 0 && smx > 0.f) atomicMax(&a.ws.smax2[b], __float_as_uint(smx));
}

// Exact top-k over the scored positions (the Full layer's candidates, or a Reindex pool).
template <int BLOCK>
__global__ void __launch_bounds__(kSelCta) select_positions_kernel(const __grid_constant__ IdxArgs a) {
  extern __shared__ __align__(16) float s_pv[];
  __shared__ uint32_t s_hist[kHistBins];
  __shared__ uint32_t s_flag[kFlagWords];
  __shared__ int32_t s_unc_id[kUncSmem];
  __shared__ float2 s_unc_val[kUncSmem];
  __shared__ int32_t s_lut[256];
  __shared__ int s_cnt[8];
  __shared__ int s_scan[72];
  __shared__ int s_out[4];
  __shared__ double s_E;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const SeqTable e = seq_entry(a.c, b, a.max_len, nullptr);
  const int32_t *list;
  int count;
  if (a.use_pool) { list = a.pool_in + (int64_t)b * a.n_keep; count = a.n_keep; }
  else { list = a.ws.pcb + (int64_t)b * a.n_keep; count = (int)a.ws.pcb_cnt[b]; }
  const int n = count * BLOCK;
  const float *pv_g = a.ws.pvals + (int64_t)b * a.n_keep * BLOCK;
  const bool staged = n <= kPvalSmem;
  if (staged)
    for (int i = tid; i < n; i += blockDim.x) s_pv[i] = __ldcg(pv_g + i);
  if (a.use_pool)
    for (int i = tid + 1; i < count; i += blockDim.x) {
      const int32_t v = __ldg(list + i);
      if (v >= 0 && __ldg(list + i - 1) >= v) set_err(a.d_err, CSA2_DEVERR_POOL);   // the pool must ascend
    }
  fill_e4m3_lut(s_lut);
  if (warp == 0) {
    double E = seq_bound(a.q + (int64_t)b * kHIdx * kDIdx, a.w + (int64_t)b * kHIdx, __uint_as_float(a.ws.smax2[b]),
                         lane);
    if (lane == 0) s_E = E;
  }
  __syncthreads();
  SelSmem sm{s_hist, s_flag, s_unc_id, s_unc_val, s_cnt, s_scan, s_out, s_lut};
  select_topk<BLOCK>(a, e, b, list, n, staged ? s_pv : pv_g, s_E, a.topk_out + (int64_t)b * a.topk, sm);
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
  const int64_t unc = nbm + (nbm > npos ? nbm : npos);
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
  w.unc_cap = nbm + (nbm > npos ? nbm : npos);
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
  w.unc_val = (float2 *)p;
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

static size_t scan_smem_bytes(int B) { return kScanSmem + (size_t)(2 * B + 1) * 8 + (size_t)B * 4; }

// persistent scan grid: every resident CTA slot of the GPU, capped by the work
template <int BLOCK>
static int scan_grid_size(int B, int64_t max_len) {
  static int per_sm = 0, for_b = -1;
  if (for_b != B) {
    const size_t smem = scan_smem_bytes(B);
    cudaFuncSetAttribute(scan_kernel<BLOCK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem_bytes(CSA2_MAX_B));
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, scan_kernel<BLOCK>, kScanWarps * 32, smem) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    for_b = B;
  }
  const int64_t units_ub = (int64_t)B * ((max_len + 15) / 16);
  const int64_t g = std::min<int64_t>((units_ub + kScanWarps - 1) / kScanWarps, (int64_t)num_sms() * per_sm);
  return (int)std::max<int64_t>(g, 1);
}

template <int BLOCK>
static void select_smem_optin() {
  static bool done = false;
  if (!done) {
    cudaFuncSetAttribute(finalize_blocks_kernel<BLOCK>, cudaFuncAttributeMaxDynamicSharedMemorySize, kCandSmem * 8);
    cudaFuncSetAttribute(select_positions_kernel<BLOCK>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPvalSmem * 4);
    done = true;
  }
}

static int positions_grid(int B) { return std::max(1, std::min(32, (int)((int64_t)num_sms() * 2 / std::max(B, 1)))); }

template <int BLOCK>
static cudaError_t full_select_impl(IdxArgs &a, int64_t max_len, const csa2_profile *prof, cudaStream_t st) {
  const int B = a.c.B;
  select_smem_optin<BLOCK>();
  const int scan_grid = scan_grid_size<BLOCK>(B, max_len);
  // inside stream capture a timing event must be an external record node
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (prof) cudaStreamIsCapturing(st, &cap);
  const unsigned ev_flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  if (prof) cudaEventRecordWithFlags((cudaEvent_t)prof->start, st, ev_flags);
  scan_kernel<BLOCK><<<scan_grid, kScanWarps * 32, scan_smem_bytes(B), st>>>(a);
  if (prof) cudaEventRecordWithFlags((cudaEvent_t)prof->stop, st, ev_flags);
  const int64_t nbm = a.ws.nbm;
  dim3 cg((unsigned)((nbm + kCollectPer - 1) / kCollectPer), (unsigned)B);
  collect_kernel<BLOCK><<<cg, 256, 0, st>>>(a);
  finalize_blocks_kernel<BLOCK><<<B, kSelCta, kCandSmem * 8, st>>>(a);
  score_positions_kernel<BLOCK><<<dim3(positions_grid(B), B), 256, 0, st>>>(a);
  select_positions_kernel<BLOCK><<<B, kSelCta, kPvalSmem * 4, st>>>(a);
  return cudaGetLastError();
}

template <int BLOCK>
static cudaError_t reindex_impl(IdxArgs &a, cudaStream_t st) {
  const int B = a.c.B;
  select_smem_optin<BLOCK>();
  score_positions_kernel<BLOCK><<<dim3(positions_grid(B), B), 256, 0, st>>>(a);
  select_positions_kernel<BLOCK><<<B, kSelCta, kPvalSmem * 4, st>>>(a);
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
  scan_kernel<8><<<scan_grid_size<8>(B, max_len), kScanWarps * 32, scan_smem_bytes(B), st>>>(a);
  bound_kernel<<<B, 32, 0, st>>>(a, bound);
  return cudaGetLastError();
}

}  // namespace csa2
