// sparse_attn_decode: gathered FP4 dequantisation fused into one softmax over the
// selected global rows plus the FP8 sliding window (V = K).
//
// Method: ttj.kr "DeepSeek-V4.1-Flash, KV 캐시를 토큰당 890바이트까지 압축하다", section
// "CSA2와 어텐션 재설계" (128-token local window combined with global sparse retrieval);
// origotech.dev deep dive, subsection "Compressed Sparse Attention 2(CSA2)" (top-k 512).
//
// A cluster of `split` CTAs per (query row, group of 16 heads) shares the row's tiles:
// each warp of each CTA owns a contiguous run of 16-row tiles and streams their raw rows
// (packed FP4 codes + E4M3 group scales, or FP8 window rows + their float32 scale) through
// a kAttnRing-slot cp.async ring, so every gather of the warp is in flight before the
// first tile is computed.  A tile is dequantised exactly to f16 in shared memory and
// consumed by mma.sync: S = Q K^T (M = 16 heads), online softmax in f32, O += P V with P
// split into f16 hi + lo parts (P V error ~2^-22).  Warps merge (m, l, O) through padded
// shared-memory slices; then every CTA of the cluster sends each slice of output dims of
// its partial O to the CTA that owns those dims, and its (m, l) to all, through
// distributed shared memory; each CTA merges and writes its dims of the row.
// Short batches of rows use larger clusters so that the whole GPU takes part.  Nothing is
// allocated and no CTA waits on a CTA outside its cluster.
//
// Exactness of the operands: an E2M1 value times its E4M3 group scale has at most 6
// significant bits within [2^-10, 2688] and is exact in f16; an E4M3 value is exact in
// f16 (the window's float32 row scale is applied to the scores and to P instead).
#include <cfloat>

#include "common.cuh"
#include "launch.h"

namespace csa2 {

#ifndef CSA2_ATTN_WARPS
#define CSA2_ATTN_WARPS 8
#endif
constexpr int kAttnWarps = CSA2_ATTN_WARPS;
constexpr int kTileRows = 16;
constexpr int kStride = 136;          // halfs per f16 tile row: 128 + 8 (conflict-free ldmatrix)
constexpr int kSlot = 2112;           // raw tile: FP4 16 x (64 + 8) = 1,152 B; FP8 16 x 128 + 16 x 4 = 2,112 B
constexpr int kAttnRing = 4;          // raw tile slots per warp
constexpr int kOStride = 132;         // floats per merge-slice row
constexpr int kMaxSplit = 8;           // CTAs per cluster (portable maximum)
constexpr int kRecvFloats = 16 * kD + 2 * 16 * kMaxSplit;          // received partial slices + (m, l)
constexpr int kTileBytes = kTileRows * kStride * 2;                 // 4,352 B
constexpr int kRingBytes = kAttnRing * kSlot;                       // 8,448 B (= 16 x 132 x 4)
constexpr float kLog2e = 1.4426950408889634f;
static_assert(kRingBytes >= 16 * kOStride * 4, "merge slice must fit in a warp's ring");

struct AttnArgs {
  csa2_cache c;
  csa2_swa swa;
  const uint16_t *q;
  int H;
  int64_t T;
  const int32_t *q_seq;
  const int64_t *q_pos;
  const int32_t *topk_idx;
  int topk, window;
  float tau;
  float *out, *lse;
  int tiles_sel, tiles_win;
  int split;              // CTAs per cluster sharing one row's tiles
  int32_t *d_err;
};

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ void sts128(uint16_t *dst, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4 *>(dst) = make_uint4(a, b, c, d);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// shared address of the same variable in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;\n" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__global__ void __launch_bounds__(kAttnWarps * 32) attn_decode_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ __align__(16) uint8_t s_dyn[];
  __shared__ __align__(16) uint16_t s_q[16 * kStride];
  __shared__ float s_rs[kAttnWarps][kTileRows], s_vs[kAttnWarps][kTileRows];
  __shared__ uint32_t s_vmask[kAttnWarps][kAttnRing];
  __shared__ float s_m[kAttnWarps][16], s_l[kAttnWarps][16];
  __shared__ float s_cm[16], s_cl[16];

  pdl_enter();
  const int split = a.split;
  const int t = blockIdx.x / split, hg = blockIdx.y;
  const int crank = split > 1 ? (int)cluster_rank() : 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;
  uint16_t *tile = reinterpret_cast<uint16_t *>(s_dyn + warp * kTileBytes);
  uint8_t *ring = s_dyn + kAttnWarps * kTileBytes + warp * kRingBytes;
  // received partials: O slices [split][16][128 / split], then m [split][16], l [split][16]
  float *s_recv = reinterpret_cast<float *>(s_dyn + kAttnWarps * (kTileBytes + kRingBytes));
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
  // every CTA of the cluster has started before any writes into another's shared memory
  if (split > 1) cluster_arrive_relaxed();

  // ---- the query row, its sequence and this warp's first indices, loaded together
  const int slots = split * kAttnWarps, slot_id = crank * kAttnWarps + warp;
  const int n_tiles_max = a.tiles_sel + a.tiles_win;
  const int tw0 = (int)((int64_t)n_tiles_max * slot_id / slots);
  const int tw1_max = (int)((int64_t)n_tiles_max * (slot_id + 1) / slots);
  const int r = lane >> 1, hf = lane & 1;
  const int32_t *idx_row = a.topk_idx + (int64_t)t * a.topk;
  int32_t idx_pre[kAttnRing];
#pragma unroll
  for (int s = 0; s < kAttnRing; ++s) {
    const int ti = tw0 + s, j = ti * kTileRows + r;
    idx_pre[s] = (ti < tw1_max && ti < a.tiles_sel && j < a.topk) ? __ldg(idx_row + j) : -1;
  }
  // the row's sequence, and its base and length: for up to 128 sequences every lane also
  // loads four table entries at once, so the entry of the row's sequence comes by shuffle
  // instead of a second dependent load
  const int b = a.q_seq[t];
  const int64_t p = a.q_pos[t];
  int64_t tb[4];
  int32_t tl[4];
  const bool small_table = a.c.B <= 128;
  if (small_table) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = lane + 32 * j;
      tb[j] = e < a.c.B ? a.c.seq_base[e] : 0;
      tl[j] = e < a.c.B ? a.c.seq_len[e] : 0;
    }
  }
  bool ok = b >= 0 && b < a.c.B;
  int64_t base = 0, len = 0;
  if (small_table) {
    const int bs = ok ? b : 0, j = bs >> 5;
    const int64_t bj = j == 0 ? tb[0] : j == 1 ? tb[1] : j == 2 ? tb[2] : tb[3];
    const int32_t lj = j == 0 ? tl[0] : j == 1 ? tl[1] : j == 2 ? tl[2] : tl[3];
    base = __shfl_sync(0xffffffffu, bj, bs & 31);
    len = __shfl_sync(0xffffffffu, lj, bs & 31);
  } else if (ok) {
    base = a.c.seq_base[b];
    len = a.c.seq_len[b];
  }
  if (ok) ok = p >= 0 && p < len && base >= 0 && base + len <= a.c.T_cap;
  if (!ok && hg == 0 && crank == 0 && tid == 0)
    set_err(a.d_err, (b < 0 || b >= a.c.B) ? CSA2_DEVERR_SEQ : CSA2_DEVERR_POS);

  // ---- queries (bf16 -> f16 into shared memory); their loads overlap the first gathers
  // 16 heads x 16 chunks of 8 values: kQPer per thread (threads beyond 256 load none)
  constexpr int kQPer = (256 + kAttnWarps * 32 - 1) / (kAttnWarps * 32);
  uint4 qv[kQPer];
#pragma unroll
  for (int j = 0; j < kQPer; ++j) {
    const int i = tid + j * kAttnWarps * 32, h = i >> 4, c8 = i & 15;
    qv[j] = i < 256 ? __ldg(reinterpret_cast<const uint4 *>(a.q + ((int64_t)t * a.H + 16 * hg + h) * kD + 8 * c8))
                    : make_uint4(0, 0, 0, 0);
  }

  // ---- this warp's tiles: the row's tiles are split evenly over every warp of the cluster
  const int tw1 = ok ? tw1_max : tw0;
  const int swa_ring = a.swa.ring;
  auto issue = [&](int ti, int slot, int32_t idx) {
    const uint32_t dst = ring_s + slot * kSlot;
    bool valid = false;
    if (ti < a.tiles_sel) {
      if (idx >= 0) {
        if (idx > p) { if (hf == 0) set_err(a.d_err, CSA2_DEVERR_INDEX); }
        else valid = true;
      }
      const int64_t row = base + (valid ? idx : 0);
      const uint8_t *src = a.c.kv_codes + row * (kD / 2) + 32 * hf;
      cp_async16(dst + r * 64 + 32 * hf, valid ? src : a.c.kv_codes, valid);
      cp_async16(dst + r * 64 + 32 * hf + 16, valid ? src + 16 : a.c.kv_codes, valid);
      cp_async4(dst + 1024 + r * 8 + 4 * hf, valid ? a.c.kv_scales + row * (kD / 16) + 4 * hf : a.c.kv_scales, valid);
    } else {
      const int j = (ti - a.tiles_sel) * kTileRows + r;
      const int64_t pj = p - a.window + 1 + j;
      valid = j < a.window && pj >= 0;
      const int64_t srow = (int64_t)b * swa_ring + (valid ? pj % swa_ring : 0);
      const uint8_t *src = a.swa.codes + srow * kD + 64 * hf;
#pragma unroll
      for (int c = 0; c < 4; ++c) cp_async16(dst + r * 128 + 64 * hf + 16 * c, valid ? src + 16 * c : a.swa.codes, valid);
      if (hf == 0) cp_async4(dst + 2048 + 4 * r, valid ? a.swa.scale + srow : a.swa.scale, valid);
    }
    const uint32_t vm = __ballot_sync(0xffffffffu, valid);
    if (lane == 0) s_vmask[warp][slot] = vm;
    cp_async_commit();
  };
#pragma unroll
  for (int s = 0; s < kAttnRing; ++s) {
    if (tw0 + s < tw1) issue(tw0 + s, s, idx_pre[s]);
    else cp_async_commit();
  }
#pragma unroll
  for (int j = 0; j < kQPer; ++j) {
    const int i = tid + j * kAttnWarps * 32, h = i >> 4, c8 = i & 15;
    if (i >= 256) break;
    const uint32_t w[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
    uint32_t o4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) o4[k] = pack_f16x2(bf16_to_f32(w[k] & 0xFFFFu), bf16_to_f32(w[k] >> 16));
    sts128(s_q + h * kStride + 8 * c8, o4[0], o4[1], o4[2], o4[3]);
  }
  __syncthreads();

  // Q fragments (A operand of S = Q K^T) through ldmatrix: heads g (a0, a2) and g + 8 (a1, a3)
  uint32_t qa[8][4];
#pragma unroll
  for (int s = 0; s < 8; ++s)
    ldsm_x4(qa[s][0], qa[s][1], qa[s][2], qa[s][3],
            s_q + ((lane >> 3) & 1) * 8 * kStride + (lane & 7) * kStride + 16 * s + 8 * (lane >> 4));

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[16][4];
#pragma unroll
  for (int d = 0; d < 16; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;

  for (int i = 0; tw0 + i < tw1; ++i) {
    const int ti = tw0 + i, slot = i % kAttnRing;
    cp_async_wait<kAttnRing - 1>();
    __syncwarp();
    const uint32_t vmask = s_vmask[warp][slot];
    const uint8_t *raw = ring + slot * kSlot;
    uint16_t *dst = tile + r * kStride + 64 * hf;
    float rs = 0.f, vs = 0.f;
    if (ti < a.tiles_sel) {
      const uint4 c0 = *reinterpret_cast<const uint4 *>(raw + r * 64 + 32 * hf);
      const uint4 c1 = *reinterpret_cast<const uint4 *>(raw + r * 64 + 32 * hf + 16);
      const uint32_t sw = *reinterpret_cast<const uint32_t *>(raw + 1024 + r * 8 + 4 * hf);
      const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      uint32_t sp[2];                                          // the four group scales as f16 pairs
      e4m3x4_to_f16(sw, sp[0], sp[1]);
#pragma unroll
      for (int gi = 0; gi < 4; ++gi) {
        const uint32_t sh = (gi & 1) ? (sp[gi >> 1] >> 16) : (sp[gi >> 1] & 0xFFFFu);
        const uint32_t s2 = sh | (sh << 16);
        uint32_t lo[4], hi[4], v[8];
        e2m1x8_to_f16(cw[2 * gi], lo);
        e2m1x8_to_f16(cw[2 * gi + 1], hi);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[k] = hmul2_u32(lo[k], s2);
          v[4 + k] = hmul2_u32(hi[k], s2);
        }
        sts128(dst + 16 * gi, v[0], v[1], v[2], v[3]);
        sts128(dst + 16 * gi + 8, v[4], v[5], v[6], v[7]);
      }
      rs = a.tau;
      vs = 1.f;
    } else {
      const float sc = *reinterpret_cast<const float *>(raw + 2048 + 4 * r);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 w = *reinterpret_cast<const uint4 *>(raw + r * 128 + 64 * hf + 16 * c);
        uint32_t v[8];
        e4m3x4_to_f16(w.x, v[0], v[1]);
        e4m3x4_to_f16(w.y, v[2], v[3]);
        e4m3x4_to_f16(w.z, v[4], v[5]);
        e4m3x4_to_f16(w.w, v[6], v[7]);
        sts128(dst + 16 * c, v[0], v[1], v[2], v[3]);
        sts128(dst + 16 * c + 8, v[4], v[5], v[6], v[7]);
      }
      rs = a.tau * sc;
      vs = sc;
    }
    if (hf == 0) { s_rs[warp][r] = rs; s_vs[warp][r] = vs; }
    __syncwarp();
    // the slot is free again: start the gather of a later tile into it
    if (tw0 + i + kAttnRing < tw1) {
      const int ti = tw0 + i + kAttnRing, j = ti * kTileRows + r;
      issue(ti, slot, ti < a.tiles_sel && j < a.topk ? __ldg(idx_row + j) : -1);
    } else {
      cp_async_commit();
    }

    // ---- S = Q K^T over the 16 rows (two n-tiles of 8 rows)
    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; s += 2) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(r0, r1, r2, r3, tile + (8 * nt + (lane & 7)) * kStride + 16 * s + 8 * (lane >> 3));
        mma_16816(sc[nt], qa[s][0], qa[s][1], qa[s][2], qa[s][3], r0, r1);
        mma_16816(sc[nt], qa[s + 1][0], qa[s + 1][1], qa[s + 1][2], qa[s + 1][3], r2, r3);
      }
    }
    // rows held by this thread: 8nt + 2tq + {0,1}; lanes 2r, 2r+1 hold row r's validity
    float z[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int row = 8 * nt + 2 * tq + k;
        const bool rv = (vmask >> (2 * row)) & 1u;
        const float f = s_rs[warp][row];
        z[nt][k] = rv ? sc[nt][k] * f : -INFINITY;
        z[nt][2 + k] = rv ? sc[nt][2 + k] * f : -INFINITY;
      }
    }
    float mx0 = fmaxf(fmaxf(z[0][0], z[0][1]), fmaxf(z[1][0], z[1][1]));
    float mx1 = fmaxf(fmaxf(z[0][2], z[0][3]), fmaxf(z[1][2], z[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = (mn0 == -INFINITY) ? 1.f : ex2_approx((m0 - mn0) * kLog2e);
    const float al1 = (mn1 == -INFINITY) ? 1.f : ex2_approx((m1 - mn1) * kLog2e);
    m0 = mn0;
    m1 = mn1;
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        pr[nt][k] = z[nt][k] == -INFINITY ? 0.f : ex2_approx((z[nt][k] - mn0) * kLog2e);
        pr[nt][2 + k] = z[nt][2 + k] == -INFINITY ? 0.f : ex2_approx((z[nt][2 + k] - mn1) * kLog2e);
      }
    }
    l0 = l0 * al0 + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
    l1 = l1 * al1 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
#pragma unroll
    for (int d = 0; d < 16; ++d) {
      o[d][0] *= al0; o[d][1] *= al0;
      o[d][2] *= al1; o[d][3] *= al1;
    }
    // P' = p * (value scale of the row), split into f16 hi + lo
    uint32_t ahi[4], alo[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float v0 = s_vs[warp][8 * nt + 2 * tq], v1 = s_vs[warp][8 * nt + 2 * tq + 1];
      const float p0 = pr[nt][0] * v0, p1 = pr[nt][1] * v1, p2 = pr[nt][2] * v0, p3 = pr[nt][3] * v1;
      const __half2 h01 = __floats2half2_rn(p0, p1), h23 = __floats2half2_rn(p2, p3);
      const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
      ahi[2 * nt] = *reinterpret_cast<const uint32_t *>(&h01);
      ahi[2 * nt + 1] = *reinterpret_cast<const uint32_t *>(&h23);
      alo[2 * nt] = pack_f16x2(p0 - f01.x, p1 - f01.y);
      alo[2 * nt + 1] = pack_f16x2(p2 - f23.x, p3 - f23.y);
    }
    // A fragment order: a0 = (head g, rows 2tq..), a1 = (head g+8, rows 2tq..),
    //                   a2 = (head g, rows 8+2tq..), a3 = (head g+8, rows 8+2tq..)
#pragma unroll
    for (int d = 0; d < 16; d += 2) {
      uint32_t r0, r1, r2, r3;
      ldsm_x4_t(r0, r1, r2, r3, tile + (((lane >> 3) & 1) * 8 + (lane & 7)) * kStride + 8 * d + 8 * (lane >> 4));
      mma_16816(o[d], ahi[0], ahi[1], ahi[2], ahi[3], r0, r1);
      mma_16816(o[d], alo[0], alo[1], alo[2], alo[3], r0, r1);
      mma_16816(o[d + 1], ahi[0], ahi[1], ahi[2], ahi[3], r2, r3);
      mma_16816(o[d + 1], alo[0], alo[1], alo[2], alo[3], r2, r3);
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // ---- merge the warps: per-head maxima, then every warp's rescaled O in its own slice
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (tq == 0) {
    s_m[warp][g] = m0; s_m[warp][g + 8] = m1;
    s_l[warp][g] = l0; s_l[warp][g + 8] = l1;
  }
  __syncthreads();
  float ms0 = -INFINITY, ms1 = -INFINITY;
#pragma unroll
  for (int w = 0; w < kAttnWarps; ++w) { ms0 = fmaxf(ms0, s_m[w][g]); ms1 = fmaxf(ms1, s_m[w][g + 8]); }
  const float f0 = (m0 == -INFINITY) ? 0.f : exp2f((m0 - ms0) * kLog2e);
  const float f1 = (m1 == -INFINITY) ? 0.f : exp2f((m1 - ms1) * kLog2e);
  float *slice = reinterpret_cast<float *>(ring);          // the ring is drained: reuse it
#pragma unroll
  for (int d = 0; d < 16; ++d) {
    const int col = 8 * d + 2 * tq;
    *reinterpret_cast<float2 *>(slice + g * kOStride + col) = make_float2(o[d][0] * f0, o[d][1] * f0);
    *reinterpret_cast<float2 *>(slice + (g + 8) * kOStride + col) = make_float2(o[d][2] * f1, o[d][3] * f1);
  }
  if (tid < 16) {
    float cm = -INFINITY, cl = 0.f;
    for (int w = 0; w < kAttnWarps; ++w) cm = fmaxf(cm, s_m[w][tid]);
    for (int w = 0; w < kAttnWarps; ++w)
      cl += (s_m[w][tid] == -INFINITY) ? 0.f : s_l[w][tid] * exp2f((s_m[w][tid] - cm) * kLog2e);
    s_cm[tid] = cm;
    s_cl[tid] = cl;
  }
  __syncthreads();
  const int64_t head0 = (int64_t)t * a.H + 16 * hg;
  const uint8_t *rings = s_dyn + kAttnWarps * kTileBytes;
  if (split == 1) {
    for (int i = tid; i < 16 * 32; i += blockDim.x) {       // 4 consecutive dims per thread
      const int h = i >> 5, d4 = (i & 31) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        const float4 v = *reinterpret_cast<const float4 *>(rings + w * kRingBytes + (h * kOStride + d4) * 4);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      const float l = s_cl[h];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      *reinterpret_cast<float4 *>(a.out + (head0 + h) * kD + d4) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    if (a.lse && tid < 16) a.lse[head0 + tid] = s_cl[tid] > 0.f ? s_cm[tid] + logf(s_cl[tid]) : -INFINITY;
    return;
  }
  // ---- cluster merge: CTA q owns output dims [q * dw, (q + 1) * dw); every CTA sends it
  // that slice of its partial O and sends its (m, l) to every CTA
  const int dw = kD / split;
  cluster_wait_acquire();                                      // every CTA of the cluster is running
  const uint32_t recv_s = (uint32_t)__cvta_generic_to_shared(s_recv);
  for (int i = tid; i < 16 * 32; i += blockDim.x) {
    const int h = i >> 5, d4 = (i & 31) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float4 v = *reinterpret_cast<const float4 *>(rings + w * kRingBytes + (h * kOStride + d4) * 4);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    const int owner = d4 / dw;
    st_cluster_v4(map_to_rank(recv_s + ((crank * 16 + h) * dw + (d4 - owner * dw)) * 4, (uint32_t)owner), acc);
  }
  for (int i = tid; i < 16 * split; i += blockDim.x) {
    const int owner = i >> 4, h = i & 15;
    const uint32_t at = map_to_rank(recv_s + (16 * kD + crank * 16 + h) * 4, (uint32_t)owner);
    st_cluster_f32(at, s_cm[h]);
    st_cluster_f32(at + 16 * kMaxSplit * 4, s_cl[h]);
  }
  cluster_arrive_release();
  cluster_wait_acquire();
  const float *rm = s_recv + 16 * kD, *rl = rm + 16 * kMaxSplit;
  if (tid < 16) {
    float M = -INFINITY, L = 0.f;
    for (int q = 0; q < split; ++q) M = fmaxf(M, rm[q * 16 + tid]);
    for (int q = 0; q < split; ++q) {
      const float mq = rm[q * 16 + tid];
      L += mq == -INFINITY ? 0.f : rl[q * 16 + tid] * exp2f((mq - M) * kLog2e);
    }
    s_cm[tid] = M;
    s_cl[tid] = L;
  }
  __syncthreads();
  for (int i = tid; i < 16 * (dw / 4); i += blockDim.x) {
    const int h = i / (dw / 4), d4 = (i % (dw / 4)) * 4;
    const float M = s_cm[h];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < split; ++q) {
      const float mq = rm[q * 16 + h];
      const float f = mq == -INFINITY ? 0.f : exp2f((mq - M) * kLog2e);
      const float4 v = *reinterpret_cast<const float4 *>(s_recv + (q * 16 + h) * dw + d4);
      acc.x += v.x * f; acc.y += v.y * f; acc.z += v.z * f; acc.w += v.w * f;
    }
    const float l = s_cl[h];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    *reinterpret_cast<float4 *>(a.out + (head0 + h) * kD + crank * dw + d4) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (crank == 0 && a.lse && tid < 16) a.lse[head0 + tid] = s_cl[tid] > 0.f ? s_cm[tid] + logf(s_cl[tid]) : -INFINITY;
}

// ------------------------------------------------------------------ host side

static size_t attn_smem(int split) {
  return (size_t)kAttnWarps * (kTileBytes + kRingBytes) + (split > 1 ? (size_t)kRecvFloats * 4 : 0);
}

size_t attn_ws_bytes(int64_t, int32_t, int32_t, int32_t) { return 0; }

// CTAs per cluster: the largest power of two (<= 8) that keeps every (row, head group)
// cluster resident at once (CSA2_ATTN_CTAS_PER_SM CTAs per SM).
#ifndef CSA2_ATTN_CTAS_PER_SM
#define CSA2_ATTN_CTAS_PER_SM 1
#endif
#ifndef CSA2_ATTN_MAX_SPLIT
#define CSA2_ATTN_MAX_SPLIT kMaxSplit
#endif
static int attn_split(int64_t rows) {
  int split = 1;
  while (split < CSA2_ATTN_MAX_SPLIT && rows * split * 2 <= CSA2_ATTN_CTAS_PER_SM * (int64_t)num_sms()) split *= 2;
  return split;
}

cudaError_t launch_attn_decode(const csa2_cache &c, const csa2_swa &swa, const uint16_t *q, int H, int64_t T,
                               const int32_t *q_seq, const int64_t *q_pos, const int32_t *topk_idx, int topk,
                               int window, float tau, float *out, float *lse, void *, int32_t *d_err,
                               cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (attn_tc_eligible(T, H) && topk + window > 0)
    return launch_attn_chunked_tc(c, swa, q, H, T, q_seq, q_pos, topk_idx, topk, window, tau, out, lse, d_err, st);
  opt_in_smem((const void *)attn_decode_kernel, attn_smem(kMaxSplit), kSiteAttnOptin, 0);
  AttnArgs a;
  a.c = c; a.swa = swa; a.q = q; a.H = H; a.T = T; a.q_seq = q_seq; a.q_pos = q_pos;
  a.topk_idx = topk_idx; a.topk = topk; a.window = window; a.tau = tau; a.out = out; a.lse = lse;
  a.d_err = d_err;
  a.tiles_sel = (topk + kTileRows - 1) / kTileRows;
  a.tiles_win = (window + kTileRows - 1) / kTileRows;
  a.split = attn_split(T * (H / 16));
  return launch_k(attn_decode_kernel, dim3((unsigned)(T * a.split), (unsigned)(H / 16)), dim3(kAttnWarps * 32),
                  attn_smem(a.split), st, (unsigned)a.split, a);
}

}  // namespace csa2
