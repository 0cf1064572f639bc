// Chunked-query indexer scores on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Method: the Full layer's indexer score (origotech.dev deep dive, subsection "Compressed
// Sparse Attention 2(CSA2)"), sigma_t = s_t * sum_h w_h * max(q_h . k_t, 0), for many query
// rows of one session at once.  Thirty-two rows share every key, so their 32 x 8 head
// queries form the N = 256 side of one dense contraction per tile of 128 keys:
//   D = K Q^T      (M = 128 keys, N = 32 rows x 8 heads, K = 64 dims)
// The E4M3 keys are converted exactly to f16 into shared-memory core matrices, the queries
// are scaled per (row, head) by the same power of two as in the one-query scan (so the same
// certified error bound holds), D accumulates in TMEM, and the epilogue (thread <-> key,
// eight rows per thread in two passes of four) forms ReLU * w summed over the heads with
// packed f32x2 FMAs, applies the key scale, stores every position's score for the exact
// selection that follows, and takes the block maxima by a reduce-scatter across the lanes
// of each block (each lane ends with whole rows' maxima) for their histogram.  A row only
// counts the positions up to its own (its length in the row view); tiles that every row of
// a warp reaches past skip the per-position checks.
//
// Pipeline per CTA (persistent over (group, tile) items): the raw bytes of the next tile
// are loaded into registers while the current tile is converted, one thread issues the
// MMAs into one of two TMEM accumulators, and the epilogue of the previous tile runs while
// the tensor cores work on the current one.
#include <cfloat>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace csa2 {

constexpr int kCqRows = 32;                                // query rows per group
constexpr int kCqKeys = 128;                               // keys per tile (MMA M)
constexpr int kCqN = kCqRows * kHIdx;                      // MMA N = 256
constexpr int kCqThreads = 512;                            // 16 warps: 4 per TMEM lane quarter
constexpr int kCqCols = 2 * kCqN;                          // TMEM: two accumulators
constexpr int kCqTileBytes = kCqKeys * kDIdx * 2;          // 16 KB of f16 keys
constexpr int kCqQ = 0;                                    // Q: 256 x 64 f16, 32 KB
constexpr int kCqK = kCqQ + kCqN * kDIdx * 2;              // two key tiles
constexpr int kCqSmem = kCqK + 2 * kCqTileBytes;           // 64 KB
constexpr int kCqSmemLaunch = 96 * 1024;                   // one CTA per SM (also set by its registers and TMEM)
constexpr int kCqMaxGroups = CSA2_MAX_B / kCqRows;
constexpr int kCqRowGroupBytes = (kDIdx / 8) * 128;        // 8 rows x 64 dims: 8 core matrices
static_assert(kCqSmem <= kCqSmemLaunch, "layout");
static_assert(kCqN == 256, "one accumulator is 256 columns");

// Byte offset of (row n, dims 8kg..8kg+7) in a K-major no-swizzle operand of 64 dims.
__device__ __forceinline__ int cq_off(int n, int kg) { return (n >> 3) * kCqRowGroupBytes + kg * 128 + (n & 7) * 16; }

// d = a * b + c on two float32 lanes at once, each rounded to nearest
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  const uint64_t ab = ((uint64_t)__float_as_uint(a.y) << 32) | __float_as_uint(a.x);
  const uint64_t bb = ((uint64_t)__float_as_uint(b.y) << 32) | __float_as_uint(b.x);
  const uint64_t cb = ((uint64_t)__float_as_uint(c.y) << 32) | __float_as_uint(c.x);
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(r) : "l"(ab), "l"(bb), "l"(cb));
  return make_float2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}

// A group of rows is scored here when all its rows share one session (one base).
__device__ __forceinline__ bool cq_uniform(const CqArgs &a, int g, int64_t &base, int32_t &maxlen) {
  const int r0 = g * kCqRows, r1 = min(a.n, r0 + kCqRows);
  base = a.base_v[r0];
  maxlen = 0;
  bool uni = true;
  for (int r = r0; r < r1; ++r) {
    uni = uni && a.base_v[r] == base;
    maxlen = max(maxlen, a.len_v[r]);
  }
  return uni;
}

template <int BLOCK>
__global__ void __launch_bounds__(kCqThreads, 1) chunk_scores_tc_kernel(const __grid_constant__ CqArgs a) {
  extern __shared__ __align__(1024) uint8_t s_dyn[];
  __shared__ __align__(8) uint64_t s_mbar[2];
  __shared__ uint32_t s_tmem;
  __shared__ int64_t s_first[kCqMaxGroups + 1];              // first item of each group
  __shared__ int64_t s_base[kCqMaxGroups];
  __shared__ int32_t s_maxlen[kCqMaxGroups];
  __shared__ __align__(16) float s_wi[kCqRows][kHIdx];       // w * 2^-c of the current group
  __shared__ __align__(16) int32_t s_len[kCqRows];            // lengths of the current group's rows
  pdl_enter();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ngroups = (a.n + kCqRows - 1) / kCqRows;

  // ---- items: (group, tile), group-major; a group that is not uniform has none
  if (tid < ngroups) {
    int64_t base;
    int32_t ml;
    const bool uni = cq_uniform(a, tid, base, ml);
    s_base[tid] = base;
    s_maxlen[tid] = uni ? ml : 0;
  }
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_addr(&s_mbar[0])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_addr(&s_mbar[1])));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  if (tid == 0) {
    int64_t run = 0;
    for (int g = 0; g < ngroups; ++g) { s_first[g] = run; run += (s_maxlen[g] + kCqKeys - 1) / kCqKeys; }
    s_first[ngroups] = run;
  }
  __syncthreads();
  const int64_t total = s_first[ngroups];
  const int64_t it0 = total * blockIdx.x / gridDim.x, it1 = total * (blockIdx.x + 1) / gridDim.x;
  if (it0 >= it1) return;                                     // uniform across the CTA

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(&s_tmem)),
                 "r"(kCqCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t idesc = umma_idesc(kCqKeys, kCqN, 0, 0);
  uint8_t *qs = s_dyn + kCqQ;
  const uint32_t qs_a = smem_addr(qs), ks_a = smem_addr(s_dyn + kCqK);

  // item cursors (group, tile): one for the tile being issued, one for the loads ahead
  int g_it, g_ft;
  int64_t t_it, t_ft;
  {
    int lo = 0, hi = ngroups;                                   // s_first[lo] <= it0 < s_first[lo + 1]
    while (hi - lo > 1) { const int mid = (lo + hi) >> 1; if (s_first[mid] <= it0) lo = mid; else hi = mid; }
    while (s_first[lo + 1] == s_first[lo]) ++lo;
    g_it = g_ft = lo;
    t_it = t_ft = it0 - s_first[lo];
  }
  auto advance = [&](int &g, int64_t &t) {
    if (++t == s_first[g + 1] - s_first[g]) {
      t = 0;
      do { ++g; } while (g < ngroups && s_first[g + 1] == s_first[g]);
    }
  };

  // converter role: key km of a tile, dims 16 dq .. 16 dq + 15; the same thread runs the
  // epilogue of key km for rows 4 eq .. 4 eq + 3 of the group (TMEM columns 32 eq ..)
  const int km = tid & (kCqKeys - 1), dq = tid >> 7;
  const int eq = warp >> 2;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  uint4 x0 = make_uint4(0, 0, 0, 0);                         // raw codes of the next tile's key
  float xs = 0.f;                                             // its scale (0: beyond every row)
  auto fetch = [&]() {                                        // the tile at the load cursor
    const int64_t kk = t_ft * kCqKeys + km;
    const bool v = kk < s_maxlen[g_ft];
    const int64_t row = s_base[g_ft] + (v ? kk : 0);
    x0 = v ? ld_nc16(a.ik_codes + row * kDIdx + 16 * dq) : make_uint4(0, 0, 0, 0);
    xs = v ? __ldg(a.ik_scale + row) : 0.f;
  };

  // the current group's rows of this thread (8 eq .. 8 eq + 7): largest valid key scale seen
  // (smx_all: the same for every row, from the tiles that all eight rows cover)
  float smx[8], smx_all = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) smx[j] = 0.f;
  int cur_g = -1;
  auto flush_smax = [&]() {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float m = warp_max(fmaxf(smx[j], smx_all));
      const int r = cur_g * kCqRows + 8 * eq + j;
      if (lane == 0 && r < a.n && m > 0.f) atomicMax(&a.ws.smax[r], __float_as_uint(m));
      smx[j] = 0.f;
    }
    smx_all = 0.f;
  };

  uint32_t ph0 = 0, ph1 = 0;
  bool dead = false;                                          // a wait ran out (uniform after a CTA vote)
  // the pending epilogue: its tile, buffer and key scale
  bool pend = false;
  int64_t pend_tile = 0;
  int pend_buf = 0;
  float pend_ks = 0.f;
  auto epilogue = [&]() {
    const uint32_t mb = smem_addr(&s_mbar[pend_buf]);
    // warp-uniform: the TMEM load below needs every lane of the warp
    const bool ok = __all_sync(0xffffffffu, mbar_wait(mb, pend_buf ? ph1 : ph0));
    if (pend_buf) ph1 ^= 1u; else ph0 ^= 1u;
    tc_fence_after();
    if (!ok) { dead = true; if (lane == 0) set_err(a.d_err, CSA2_DEVERR_TIMEOUT); return; }
    const int em = 32 * (warp & 3) + lane;                    // == km
    const int kk = (int)pend_tile * kCqKeys + em;             // < 2^31: positions of one row
    // the warp's eight rows all reach past the tile's last key (the usual case): no
    // per-position validity (warp-uniform, as eq is)
    const int4 la = *reinterpret_cast<const int4 *>(&s_len[8 * eq]);
    const int4 lb = *reinterpret_cast<const int4 *>(&s_len[8 * eq + 4]);
    const int minlen = min(min(min(la.x, la.y), min(la.z, la.w)), min(min(lb.x, lb.y), min(lb.z, lb.w)));
    const bool full = (int)pend_tile * kCqKeys + kCqKeys <= minlen;
    float *sig = a.ws.sigma + ((int64_t)cur_g * kCqRows + 8 * eq) * a.ws.sigma_stride + kk;
    const int64_t sst = a.ws.sigma_stride;
    float blk[8];                                             // row j's score, 0 where not valid
    auto rows = [&](auto full_t) {
      constexpr bool kFull = decltype(full_t)::value;
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {                  // rows 8 eq + 4 pass + j
        float v[32];
        tmem_ld32(tmem + lane_off + pend_buf * kCqN + 64 * eq + 32 * pass, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int jj = 4 * pass + j, jr = 8 * eq + jj;
          const float4 w0 = *reinterpret_cast<const float4 *>(&s_wi[jr][0]);
          const float4 w1 = *reinterpret_cast<const float4 *>(&s_wi[jr][4]);
          // sum_h w_h max(v_h, 0) as two interleaved chains of four (w >= 0: every term is
          // non-negative, so each result keeps at most five roundings of the sum)
          float2 acc = fma2(make_float2(fmaxf(v[8 * j], 0.f), fmaxf(v[8 * j + 1], 0.f)), make_float2(w0.x, w0.y),
                            make_float2(0.f, 0.f));
          acc = fma2(make_float2(fmaxf(v[8 * j + 2], 0.f), fmaxf(v[8 * j + 3], 0.f)), make_float2(w0.z, w0.w), acc);
          acc = fma2(make_float2(fmaxf(v[8 * j + 4], 0.f), fmaxf(v[8 * j + 5], 0.f)), make_float2(w1.x, w1.y), acc);
          acc = fma2(make_float2(fmaxf(v[8 * j + 6], 0.f), fmaxf(v[8 * j + 7], 0.f)), make_float2(w1.z, w1.w), acc);
          float o = (acc.x + acc.y) * pend_ks;
          o = o > 0.f ? o : 0.f;                              // also maps NaN and -0 to +0
          const bool valid = kFull || kk < s_len[jr];
          // streaming store (evict first): 4 bytes per (row, position), read back only for
          // the candidate blocks, so the keys of the group stay in L2
          if (valid) __stcs(sig + jj * sst, o);
          if (!kFull) smx[jj] = fmaxf(smx[jj], valid ? pend_ks : 0.f);
          blk[jj] = valid ? o : 0.f;
        }
      }
    };
    if (full) { rows(std::true_type{}); smx_all = fmaxf(smx_all, pend_ks); }
    else rows(std::false_type{});

    // Block maxima by a reduce-scatter over the lanes of each block: stage s halves the
    // rows a lane holds, the lane with bit d = kBl / 2^(s+1) set keeping the upper half, so
    // lane i of a block (i < kBl) ends with the maxima of rows kNb i .. kNb i + kNb - 1.
    constexpr int kBl = BLOCK < 8 ? BLOCK : 8;
    constexpr int kNb = 8 / kBl;
    constexpr int kStages = kBl == 8 ? 3 : kBl == 4 ? 2 : kBl == 2 ? 1 : 0;
#pragma unroll
    for (int st = 0; st < kStages; ++st) {
      const int d = kBl >> (st + 1), half = 4 >> st;
      const bool up = (lane & d) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float keep = up ? blk[half + i] : blk[i];
        const float send = up ? blk[i] : blk[half + i];
        blk[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, d));
      }
    }
#pragma unroll
    for (int d = 8; d < BLOCK; d <<= 1) blk[0] = fmaxf(blk[0], __shfl_xor_sync(0xffffffffu, blk[0], d));
    // a block is recorded when its first position is valid for the row
    if ((em & (BLOCK - 1)) < kBl) {
      const int kb0 = kk & ~(BLOCK - 1);
#pragma unroll
      for (int i = 0; i < kNb; ++i) {
        const int jr = 8 * eq + (em & (kBl - 1)) * kNb + i;
        if (kb0 < s_len[jr]) {
          const int64_t r = (int64_t)cur_g * kCqRows + jr;
          a.ws.bmax[r * a.ws.nbm + kk / BLOCK] = blk[i];
          atomicAdd(&a.ws.hist[r * kHistBins + min(__float_as_uint(blk[i]) >> kHistShift, (uint32_t)kHistBins - 1)],
                    1u);
        }
      }
    }
  };

  fetch();
  advance(g_ft, t_ft);
  for (int64_t it = it0; it < it1; ++it) {
    const int g = g_it;
    const int64_t tile = t_it;
    const int buf = (int)((it - it0) & 1);
    const bool newg = g != cur_g;
    if (newg) {
      // the previous group's last tile completes before its queries are replaced
      if (pend) { epilogue(); pend = false; }
      if (cur_g >= 0) flush_smax();
      if (__syncthreads_or(dead)) break;
      // queries of group g: (row jr, head h) = MMA column n = 8 jr + h; four threads per pair,
      // two pairs per thread
#pragma unroll
      for (int pit = 0; pit < kCqN / (kCqThreads / 4); ++pit) {
        const int pair = (tid >> 2) + (kCqThreads / 4) * pit, part = tid & 3;
        const int jr = pair >> 3, h = pair & 7;
        const int r = g * kCqRows + jr;
        const bool rv = r < a.n;
        uint32_t wq[8];
        if (rv) {
          const uint4 *src = reinterpret_cast<const uint4 *>(a.q + ((int64_t)r * kHIdx + h) * kDIdx + 16 * part);
          const uint4 u0 = __ldg(src), u1 = __ldg(src + 1);
          wq[0] = u0.x; wq[1] = u0.y; wq[2] = u0.z; wq[3] = u0.w;
          wq[4] = u1.x; wq[5] = u1.y; wq[6] = u1.z; wq[7] = u1.w;
        } else {
  #pragma unroll
          for (int i = 0; i < 8; ++i) wq[i] = 0u;
      }
      float mx = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        mx = fmaxf(mx, fmaxf(fabsf(bf16_to_f32(wq[i] & 0xFFFFu)), fabsf(bf16_to_f32(wq[i] >> 16))));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const int c = head_shift(mx);
      const float sc = pow2f(c);
#pragma unroll
      for (int i = 0; i < 2; ++i) {                           // dims 16 part + 8 i .. + 7
        uint32_t o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t wv = wq[4 * i + e];
          o4[e] = pack_f16x2(bf16_to_f32(wv & 0xFFFFu) * sc, bf16_to_f32(wv >> 16) * sc);
        }
        *reinterpret_cast<uint4 *>(qs + cq_off(pair, 2 * part + i)) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      if (part == 0) s_wi[jr][h] = rv ? __ldg(a.w + (int64_t)r * kHIdx + h) * pow2f(-c) : 0.f;
      }
      if (tid < kCqRows) s_len[tid] = (g * kCqRows + tid < a.n) ? a.len_v[g * kCqRows + tid] : 0;
      cur_g = g;
    }
    // ---- this tile's keys, exactly to f16, into its buffer; then the next tile's loads
    {
      uint8_t *kb = s_dyn + kCqK + buf * kCqTileBytes;
      *reinterpret_cast<uint4 *>(kb + cq_off(km, 2 * dq)) =
          make_uint4(e4m3x2_to_f16x2(x0.x), e4m3x2_to_f16x2(x0.x >> 16), e4m3x2_to_f16x2(x0.y),
                     e4m3x2_to_f16x2(x0.y >> 16));
      *reinterpret_cast<uint4 *>(kb + cq_off(km, 2 * dq + 1)) =
          make_uint4(e4m3x2_to_f16x2(x0.z), e4m3x2_to_f16x2(x0.z >> 16), e4m3x2_to_f16x2(x0.w),
                     e4m3x2_to_f16x2(x0.w >> 16));
    }
    const float cur_ks = xs;
    if (it + 1 < it1) { fetch(); advance(g_ft, t_ft); }
    fence_async_smem();
    tc_fence_before();
    if (__syncthreads_or(dead)) break;
    tc_fence_after();
    if (tid == 0) {
      const uint32_t kb_a = ks_a + buf * kCqTileBytes;
#pragma unroll
      for (int s = 0; s < kDIdx / 16; ++s)
        umma_f16(tmem + buf * kCqN, umma_desc(kb_a + 256 * s, 128, kCqRowGroupBytes),
                 umma_desc(qs_a + 256 * s, 128, kCqRowGroupBytes), idesc, s > 0);
      umma_commit(smem_addr(&s_mbar[buf]));
    }
    __syncwarp();
    if (pend) epilogue();
    pend = true;
    pend_tile = tile;
    pend_buf = buf;
    pend_ks = cur_ks;
    advance(g_it, t_it);
  }
  dead = __syncthreads_or(dead);
  if (pend && !dead) epilogue();
  dead = __syncthreads_or(dead);
  if (cur_g >= 0 && !dead) flush_smax();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kCqCols));
}

template <int BLOCK>
static cudaError_t launch_cq(const CqArgs &a, cudaStream_t st) {
  opt_in_smem((const void *)chunk_scores_tc_kernel<BLOCK>, kCqSmemLaunch, kSiteChunkScoresOptin, BLOCK);
  return launch_k(chunk_scores_tc_kernel<BLOCK>, dim3((unsigned)num_sms()), dim3(kCqThreads), kCqSmemLaunch, st,
                  0, a);
}

cudaError_t launch_chunk_scores_tc(const CqArgs &a, int block, cudaStream_t st) {
  switch (block) {
    case 1: return launch_cq<1>(a, st);
    case 2: return launch_cq<2>(a, st);
    case 4: return launch_cq<4>(a, st);
    case 8: return launch_cq<8>(a, st);
    case 16: return launch_cq<16>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csa2
