// sparse_attn_decode: gathered FP4 dequantisation fused into one softmax over the
// selected global rows plus the FP8 sliding window (V = K).
//
// Method: ttj.kr "DeepSeek-V4.1-Flash, KV 캐시를 토큰당 890바이트까지 압축하다", section
// "CSA2와 어텐션 재설계" (128-token local window combined with global sparse retrieval);
// origotech.dev deep dive, subsection "Compressed Sparse Attention 2(CSA2)" (top-k 512).
//
// Layout of the work: one CTA per (query row, split of the KV rows, group of 16 heads);
// 4 warps per CTA, each warp owns 16-row tiles.  A tile is gathered (16-byte loads of
// packed FP4 codes + the 4 E4M3 group scales, or FP8 window rows), dequantised exactly
// to f16 into shared memory, and consumed by mma.sync: S = Q K^T (M = 16 heads), online
// softmax in f32, O += P V with P split into f16 hi + lo parts (P V error ~2^-22).
// Splits of one row merge their (m, l, O) partials in the last CTA to finish; the
// arrival counter is reset by that CTA.  Nothing waits on another CTA.
//
// Exactness of the operands: an E2M1 value times its E4M3 group scale has at most 6
// significant bits within [2^-10, 2688] and is exact in f16; an E4M3 value is exact in
// f16 (the window's float32 row scale is applied to the scores and to P instead).
#include <cfloat>

#include "common.cuh"
#include "launch.h"

namespace csa2 {

constexpr int kAttnWarps = 4;
constexpr int kTileRows = 16;
constexpr int kStride = 136;         // halfs per shared row: 128 + 8 (conflict-free ldmatrix)
constexpr float kLog2e = 1.4426950408889634f;

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
  float *part;          // [T][HG][S][16][130]: m, l, o[128]
  uint32_t *counter;    // [T][HG]
  int S, tiles_sel, tiles_win, tiles_per_split;
  int32_t *d_err;
};

constexpr int kPartStride = 130;

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  return pack_f16x2(bf16_to_f32(v & 0xFFFFu), bf16_to_f32(v >> 16));
}

__device__ __forceinline__ uint32_t fp4x2_to_f16x2(uint32_t byte) {
  __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)(byte & 0xFFu), __NV_E2M1);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

// 8 bytes of packed FP4 (16 channels of one group) times the group scale -> 8 f16x2
__device__ __forceinline__ void dequant_group(uint32_t w0, uint32_t w1, uint32_t scale_h2, uint32_t out[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = hmul2_u32(fp4x2_to_f16x2(w0 >> (8 * i)), scale_h2);
#pragma unroll
  for (int i = 0; i < 4; ++i) out[4 + i] = hmul2_u32(fp4x2_to_f16x2(w1 >> (8 * i)), scale_h2);
}

__device__ __forceinline__ void sts128(uint16_t *dst, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4 *>(dst) = make_uint4(a, b, c, d);
}

__global__ void __launch_bounds__(kAttnWarps * 32) attn_decode_kernel(const __grid_constant__ AttnArgs a) {
  __shared__ __align__(16) uint16_t s_tile[kAttnWarps][kTileRows * kStride];
  __shared__ float s_rs[kAttnWarps][kTileRows], s_vs[kAttnWarps][kTileRows];
  __shared__ float s_m[kAttnWarps][16], s_l[kAttnWarps][16];
  __shared__ float s_o[16][128];
  __shared__ int s_last;

  const int t = blockIdx.x, split = blockIdx.y, hg = blockIdx.z;
  const int HG = gridDim.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;

  // ---- the query row and its sequence
  const int b = a.q_seq[t];
  const int64_t p = a.q_pos[t];
  bool ok = b >= 0 && b < a.c.B;
  int64_t base = 0, len = 0;
  if (ok) {
    base = a.c.seq_base[b];
    len = a.c.seq_len[b];
    ok = p >= 0 && p < len && base >= 0 && base + len <= a.c.T_cap;
  }
  if (!ok && split == 0 && hg == 0 && tid == 0) set_err(a.d_err, (b < 0 || b >= a.c.B) ? CSA2_DEVERR_SEQ : CSA2_DEVERR_POS);

  // ---- Q fragments (A operand of S = Q K^T): heads 16hg+g and 16hg+g+8
  uint32_t qa[8][4];
  {
    const uint16_t *q0 = a.q + ((int64_t)t * a.H + 16 * hg + g) * kD;
    const uint16_t *q1 = q0 + 8 * kD;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int d0 = 16 * s + 2 * tq;
      qa[s][0] = bf16x2_to_f16x2(__ldg(reinterpret_cast<const uint32_t *>(q0 + d0)));
      qa[s][1] = bf16x2_to_f16x2(__ldg(reinterpret_cast<const uint32_t *>(q1 + d0)));
      qa[s][2] = bf16x2_to_f16x2(__ldg(reinterpret_cast<const uint32_t *>(q0 + d0 + 8)));
      qa[s][3] = bf16x2_to_f16x2(__ldg(reinterpret_cast<const uint32_t *>(q1 + d0 + 8)));
    }
  }

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[16][4];
#pragma unroll
  for (int d = 0; d < 16; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;

  const int n_tiles = a.tiles_sel + a.tiles_win;
  const int t0 = split * a.tiles_per_split;
  const int t1 = ok ? min(n_tiles, t0 + a.tiles_per_split) : t0;
  uint16_t *tile = s_tile[warp];
  const int swa_ring = a.swa.ring;

  for (int ti = t0 + warp; ti < t1; ti += kAttnWarps) {
    // ---- gather + dequantise 16 rows into shared memory (2 lanes per row)
    const int r = lane >> 1, hf = lane & 1;
    bool valid = false;
    float rs = 0.f, vs = 0.f;
    uint16_t *dst = tile + r * kStride + 64 * hf;
    if (ti < a.tiles_sel) {
      const int j = ti * kTileRows + r;
      int32_t idx = j < a.topk ? __ldg(a.topk_idx + (int64_t)t * a.topk + j) : -1;
      if (idx >= 0) {
        if (idx > p) {
          if (hf == 0) set_err(a.d_err, CSA2_DEVERR_INDEX);
        } else {
          valid = true;
        }
      }
      if (valid) {
        const int64_t row = base + idx;
        const uint4 c0 = ld_nc16(a.c.kv_codes + row * (kD / 2) + 32 * hf);
        const uint4 c1 = ld_nc16(a.c.kv_codes + row * (kD / 2) + 32 * hf + 16);
        const uint32_t sw = __ldg(reinterpret_cast<const uint32_t *>(a.c.kv_scales + row * (kD / 16) + 4 * hf));
        const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          const uint32_t sh = e4m3x2_to_f16x2((sw >> (8 * gi)) & 0xFFu) & 0xFFFFu;
          uint32_t v[8];
          dequant_group(cw[2 * gi], cw[2 * gi + 1], sh | (sh << 16), v);
          sts128(dst + 16 * gi, v[0], v[1], v[2], v[3]);
          sts128(dst + 16 * gi + 8, v[4], v[5], v[6], v[7]);
        }
        rs = a.tau;
        vs = 1.f;
      }
    } else {
      const int j = (ti - a.tiles_sel) * kTileRows + r;
      const int64_t pj = p - a.window + 1 + j;
      if (j < a.window && pj >= 0) {
        valid = true;
        const int64_t slot = (int64_t)b * swa_ring + (pj % swa_ring);
        const uint8_t *src = a.swa.codes + slot * kD + 64 * hf;
        const float s = __ldg(a.swa.scale + slot);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 w = ld_nc16(src + 16 * c);
          sts128(dst + 16 * c, e4m3x2_to_f16x2(w.x), e4m3x2_to_f16x2(w.x >> 16), e4m3x2_to_f16x2(w.y),
                 e4m3x2_to_f16x2(w.y >> 16));
          sts128(dst + 16 * c + 8, e4m3x2_to_f16x2(w.z), e4m3x2_to_f16x2(w.z >> 16), e4m3x2_to_f16x2(w.w),
                 e4m3x2_to_f16x2(w.w >> 16));
        }
        rs = a.tau * s;
        vs = s;
      }
    }
    if (!valid) {
#pragma unroll
      for (int c = 0; c < 8; ++c) sts128(dst + 8 * c, 0u, 0u, 0u, 0u);
    }
    if (hf == 0) { s_rs[warp][r] = rs; s_vs[warp][r] = vs; }
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
    __syncwarp();

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
    // rows held by this thread: 8nt + 2tq + {0,1}; row validity from the ballot (lanes 2r, 2r+1 hold row r)
    float z[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = 8 * nt + 2 * tq + i;
        const bool rv = (vmask >> (2 * row)) & 1u;
        const float f = s_rs[warp][row];
        z[nt][i] = rv ? sc[nt][i] * f : -INFINITY;
        z[nt][2 + i] = rv ? sc[nt][2 + i] * f : -INFINITY;
      }
    }
    float mx0 = fmaxf(fmaxf(z[0][0], z[0][1]), fmaxf(z[1][0], z[1][1]));
    float mx1 = fmaxf(fmaxf(z[0][2], z[0][3]), fmaxf(z[1][2], z[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = (mn0 == -INFINITY) ? 1.f : exp2f((m0 - mn0) * kLog2e);
    const float al1 = (mn1 == -INFINITY) ? 1.f : exp2f((m1 - mn1) * kLog2e);
    m0 = mn0;
    m1 = mn1;
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        pr[nt][i] = z[nt][i] == -INFINITY ? 0.f : exp2f((z[nt][i] - mn0) * kLog2e);
        pr[nt][2 + i] = z[nt][2 + i] == -INFINITY ? 0.f : exp2f((z[nt][2 + i] - mn1) * kLog2e);
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

  // ---- merge the 4 warps of this CTA
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (tq == 0) {
    s_m[warp][g] = m0; s_m[warp][g + 8] = m1;
    s_l[warp][g] = l0; s_l[warp][g + 8] = l1;
  }
  for (int i = tid; i < 16 * 128; i += blockDim.x) (&s_o[0][0])[i] = 0.f;
  __syncthreads();
  float ms0 = -INFINITY, ms1 = -INFINITY;
#pragma unroll
  for (int w = 0; w < kAttnWarps; ++w) { ms0 = fmaxf(ms0, s_m[w][g]); ms1 = fmaxf(ms1, s_m[w][g + 8]); }
  const float f0 = (m0 == -INFINITY) ? 0.f : exp2f((m0 - ms0) * kLog2e);
  const float f1 = (m1 == -INFINITY) ? 0.f : exp2f((m1 - ms1) * kLog2e);
  for (int w = 0; w < kAttnWarps; ++w) {
    if (warp == w) {
#pragma unroll
      for (int d = 0; d < 16; ++d) {
        const int col = 8 * d + 2 * tq;
        s_o[g][col] += o[d][0] * f0;
        s_o[g][col + 1] += o[d][1] * f0;
        s_o[g + 8][col] += o[d][2] * f1;
        s_o[g + 8][col + 1] += o[d][3] * f1;
      }
    }
    __syncthreads();
  }
  // per-head (m, l) of the CTA
  float cm = -INFINITY, cl = 0.f;
  if (tid < 16) {
    for (int w = 0; w < kAttnWarps; ++w) cm = fmaxf(cm, s_m[w][tid]);
    for (int w = 0; w < kAttnWarps; ++w)
      cl += (s_m[w][tid] == -INFINITY) ? 0.f : s_l[w][tid] * exp2f((s_m[w][tid] - cm) * kLog2e);
  }

  const int64_t head0 = (int64_t)t * a.H + 16 * hg;
  if (a.S == 1) {
    if (tid < 16) { s_m[0][tid] = cm; s_l[0][tid] = cl; }
    __syncthreads();
    for (int i = tid; i < 16 * 128; i += blockDim.x) {
      const int h = i >> 7;
      const float l = s_l[0][h];
      a.out[(head0 + h) * kD + (i & 127)] = l > 0.f ? (&s_o[0][0])[i] / l : 0.f;
    }
    if (a.lse && tid < 16) a.lse[head0 + tid] = cl > 0.f ? cm + logf(cl) : -INFINITY;
    return;
  }

  // ---- split-KV: publish this split's partial, the last CTA of the row merges
  float *mine = a.part + (((int64_t)t * HG + hg) * a.S + split) * 16 * kPartStride;
  if (tid < 16) { mine[tid * kPartStride] = cm; mine[tid * kPartStride + 1] = cl; }
  for (int i = tid; i < 16 * 128; i += blockDim.x) mine[(i >> 7) * kPartStride + 2 + (i & 127)] = (&s_o[0][0])[i];
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atomicAdd(&a.counter[(int64_t)t * HG + hg], 1u);
    s_last = (prev == (uint32_t)a.S - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float *all = a.part + ((int64_t)t * HG + hg) * a.S * 16 * kPartStride;
  if (tid < 16) {
    float M = -INFINITY, Lsum = 0.f;
    for (int s = 0; s < a.S; ++s) M = fmaxf(M, __ldcg(all + (s * 16 + tid) * kPartStride));
    for (int s = 0; s < a.S; ++s) {
      const float ms = __ldcg(all + (s * 16 + tid) * kPartStride);
      if (ms != -INFINITY) Lsum += __ldcg(all + (s * 16 + tid) * kPartStride + 1) * exp2f((ms - M) * kLog2e);
    }
    s_m[0][tid] = M;
    s_l[0][tid] = Lsum;
    if (a.lse) a.lse[head0 + tid] = Lsum > 0.f ? M + logf(Lsum) : -INFINITY;
  }
  __syncthreads();
  for (int i = tid; i < 16 * 128; i += blockDim.x) {
    const int h = i >> 7, d = i & 127;
    const float M = s_m[0][h], Lsum = s_l[0][h];
    float acc = 0.f;
    for (int s = 0; s < a.S; ++s) {
      const float ms = __ldcg(all + (s * 16 + h) * kPartStride);
      if (ms != -INFINITY) acc += __ldcg(all + (s * 16 + h) * kPartStride + 2 + d) * exp2f((ms - M) * kLog2e);
    }
    a.out[(head0 + h) * kD + d] = Lsum > 0.f ? acc / Lsum : 0.f;
  }
  if (tid == 0) a.counter[(int64_t)t * HG + hg] = 0u;
}

// ------------------------------------------------------------------ host side

static int choose_splits(int64_t T, int H, int n_tiles) {
  const int64_t ctas = T * (H / 16);
  const int64_t want = 2LL * num_sms();
  int S = (int)((want + ctas - 1) / ctas);
  const int max_s = (n_tiles + kAttnWarps - 1) / kAttnWarps;   // at least one tile per warp
  if (S > max_s) S = max_s;
  if (S < 1) S = 1;
  return S;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t attn_ws_bytes(int64_t T, int32_t H, int32_t topk, int32_t window) {
  const int n_tiles = (topk + kTileRows - 1) / kTileRows + (window + kTileRows - 1) / kTileRows;
  const int S = choose_splits(T, H, n_tiles);
  const int64_t HG = H / 16;
  if (S == 1) return 256;
  return align256((size_t)T * HG * 4) + align256((size_t)T * HG * S * 16 * kPartStride * 4);
}

cudaError_t launch_attn_decode(const csa2_cache &c, const csa2_swa &swa, const uint16_t *q, int H, int64_t T,
                               const int32_t *q_seq, const int64_t *q_pos, const int32_t *topk_idx, int topk,
                               int window, float tau, float *out, float *lse, void *ws, int32_t *d_err,
                               cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  AttnArgs a;
  a.c = c; a.swa = swa; a.q = q; a.H = H; a.T = T; a.q_seq = q_seq; a.q_pos = q_pos;
  a.topk_idx = topk_idx; a.topk = topk; a.window = window; a.tau = tau; a.out = out; a.lse = lse;
  a.d_err = d_err;
  a.tiles_sel = (topk + kTileRows - 1) / kTileRows;
  a.tiles_win = (window + kTileRows - 1) / kTileRows;
  const int n_tiles = a.tiles_sel + a.tiles_win;
  a.S = choose_splits(T, H, n_tiles);
  a.tiles_per_split = (n_tiles + a.S - 1) / a.S;
  const int64_t HG = H / 16;
  a.counter = (uint32_t *)ws;
  a.part = (float *)((char *)ws + align256((size_t)T * HG * 4));
  if (a.S > 1) {
    cudaError_t e = cudaMemsetAsync(a.counter, 0, (size_t)T * HG * 4, st);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((unsigned)T, (unsigned)a.S, (unsigned)HG);
  attn_decode_kernel<<<grid, kAttnWarps * 32, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace csa2
