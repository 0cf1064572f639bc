// Chunked-query sparse attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Method: as sparse_attn_decode (ttj.kr "DeepSeek-V4.1-Flash, KV 캐시를 토큰당 890바이트까지
// 압축하다", section "CSA2와 어텐션 재설계"; origotech.dev deep dive, subsection "Compressed
// Sparse Attention 2(CSA2)"): one softmax over a row's selected FP4 rows plus its FP8
// window, V = K.  With many query rows and 64 heads every gathered key row is shared by all
// heads of its query row, so the two products are dense contractions:
//   S^T = K Q^T      (M = 128 key rows of a chunk, N = H heads, K = 128 dims)
//   O^T += V^T P^T   (M = 128 dims,               N = H heads, K = 128 key rows)
//   l   += 1 P^T     (the row sums, from the same f16 P, on the tensor cores too)
// One CTA (8 warps) owns one query row at a time: threads k and k + 128 dequantise the two
// halves of key row k of the chunk exactly into f16 core matrices in shared memory (the
// same bytes serve as K for S and, read MN-major, as V for O), one thread issues the MMAs,
// the accumulators live in TMEM (key row / output dim k <-> TMEM lane k; the two threads of
// a lane take 32 heads each), and the softmax is online across chunks with the O and l
// accumulators rescaled in TMEM when a head's running maximum grows.
//
// Shared-memory operands use the no-swizzle core-matrix layout: 8 rows x 16 bytes per
// 128-byte core matrix; for K-major operands the descriptor's leading offset is the stride
// between core matrices along K and the stride offset the stride along M/N; for MN-major
// operands the same roles hold (leading = along K, stride = along M/N).
#include <cfloat>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace csa2 {

constexpr int kTcThreads = 256;          // 8 warps: threads k and k + 128 <-> key row k <-> TMEM lane k
constexpr int kTcChunk = 128;            // key rows per chunk (MMA M)
constexpr int kTcMaxH = 64;              // heads handled per CTA (MMA N)
constexpr int kTcCols = 256;             // TMEM columns per CTA: S | O^T | l
constexpr float kTcLog2e = 1.4426950408889634f;

// dynamic shared memory layout (bytes)
constexpr int kTcQ = 0;                                   // Q: (hg, dg) blocks, H x 128 f16   16 KB
constexpr int kTcK = kTcQ + kTcMaxH * kD * 2;             // K chunk: (kg, dg) blocks          32 KB
constexpr int kTcP = kTcK + kTcChunk * kD * 2;            // P^T: (kg, hg) blocks              16 KB
constexpr int kTcP2 = kTcP + kTcChunk * kTcMaxH * 2;      // P^T without the FP8 row scale    16 KB
constexpr int kTcOnes = kTcP2 + kTcChunk * kTcMaxH * 2;   // one core matrix of f16 ones      128 B
constexpr int kTcSmem = kTcOnes + 128;
// padding that keeps at most two CTAs on an SM (their TMEM columns fit: 2 x 256 = 512)
constexpr int kTcSmemLaunch = 96 * 1024;
static_assert(kTcSmem <= kTcSmemLaunch, "layout");

struct TcArgs {
  csa2_cache c;
  csa2_swa swa;
  const uint16_t *q;          // [T][H][128] bf16
  int H;
  int64_t T;
  const int32_t *q_seq;
  const int64_t *q_pos;
  const int32_t *topk_idx;    // [T][topk]
  int topk, window;
  float tau;
  float *out, *lse;
  int n_sel_chunks, n_chunks;
  int32_t *d_err;
};

__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;\n" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ uint32_t fp4x2_f16x2(uint32_t byte) {
  __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)(byte & 0xFFu), __NV_E2M1);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

// Half of one key row's raw bytes (dims 64h..64h+63 for thread half h), loaded ahead of
// its chunk.
struct KeyRaw {
  uint4 w[4];          // FP4: w[0..1] codes (32 B); FP8 window: w[0..3] codes (64 B)
  uint32_t sc;         // FP4: 4 E4M3 group scales
  float wsc;           // FP8: the row's float32 scale (0 for an invalid row)
  bool valid, fp8;
};

// Slot k of chunk c: the cache row it reads (via the top-k index or the window), or invalid.
__device__ __forceinline__ void key_slot(const TcArgs &a, int c, int k, int64_t t, int32_t idx_pre, bool have_pre,
                                         int64_t p, KeyRaw &kr, int64_t &row_or_pos) {
  kr.valid = false;
  kr.fp8 = c >= a.n_sel_chunks;
  kr.wsc = 0.f;                                              // invalid rows: P * scale must stay 0
  row_or_pos = -1;
  if (!kr.fp8) {
    const int j = c * kTcChunk + k;
    const int32_t idx = have_pre ? idx_pre : (j < a.topk ? __ldg(a.topk_idx + t * a.topk + j) : -1);
    if (idx >= 0 && idx > p) set_err(a.d_err, CSA2_DEVERR_INDEX);
    kr.valid = idx >= 0 && idx <= p;
    row_or_pos = idx;
  } else {
    const int j = (c - a.n_sel_chunks) * kTcChunk + k;
    const int64_t pj = p - a.window + 1 + j;
    kr.valid = j < a.window && pj >= 0;
    row_or_pos = pj;
  }
}

__device__ __forceinline__ void key_fetch(const TcArgs &a, int half, int b, int64_t base, int64_t row_or_pos,
                                          KeyRaw &kr) {
  if (!kr.valid) return;
  if (!kr.fp8) {
    const int64_t r = base + row_or_pos;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.c.kv_codes + r * (kD / 2) + 32 * half);
    kr.w[0] = __ldg(src);
    kr.w[1] = __ldg(src + 1);
    kr.sc = __ldg(reinterpret_cast<const uint32_t *>(a.c.kv_scales + r * (kD / 16) + 4 * half));
  } else {
    const int64_t srow = (int64_t)b * a.swa.ring + row_or_pos % a.swa.ring;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.swa.codes + srow * kD + 64 * half);
#pragma unroll
    for (int i = 0; i < 4; ++i) kr.w[i] = __ldg(src + i);
    kr.wsc = __ldg(a.swa.scale + srow);
  }
}

// Writes dims 64h..64h+63 of key row k of the chunk, dequantised exactly to f16, into its
// core matrices: block (k / 8, dg) holds dims 8dg..8dg+7 of keys 8(k/8)..8(k/8)+7.
__device__ __forceinline__ void store_key(uint8_t *ks, int k, int half, const KeyRaw &kr) {
  uint8_t *row = ks + (k >> 3) * 16 * 128 + (k & 7) * 16 + 8 * half * 128;
  if (!kr.valid) {
#pragma unroll
    for (int dg = 0; dg < 8; ++dg) *reinterpret_cast<uint4 *>(row + dg * 128) = make_uint4(0, 0, 0, 0);
    return;
  }
  if (!kr.fp8) {
#pragma unroll
    for (int g4 = 0; g4 < 4; ++g4) {                         // 16 channels: two core-matrix rows
      const uint32_t s16 = e4m3x2_to_f16x2((kr.sc >> (8 * g4)) & 0xFFu) & 0xFFFFu;
      const uint32_t s2 = s16 | (s16 << 16);
      const uint4 cw = kr.w[g4 >> 1];
      const uint32_t c0 = (g4 & 1) ? cw.z : cw.x, c1 = (g4 & 1) ? cw.w : cw.y;     // 8 bytes = 16 codes
      uint32_t v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = hmul2_bits(fp4x2_f16x2(c0 >> (8 * i)), s2);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[4 + i] = hmul2_bits(fp4x2_f16x2(c1 >> (8 * i)), s2);
      *reinterpret_cast<uint4 *>(row + (2 * g4) * 128) = make_uint4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<uint4 *>(row + (2 * g4 + 1) * 128) = make_uint4(v[4], v[5], v[6], v[7]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {                            // 16 codes -> two core-matrix rows
      const uint4 w = kr.w[i];
      *reinterpret_cast<uint4 *>(row + (2 * i) * 128) =
          make_uint4(e4m3x2_to_f16x2(w.x), e4m3x2_to_f16x2(w.x >> 16), e4m3x2_to_f16x2(w.y),
                     e4m3x2_to_f16x2(w.y >> 16));
      *reinterpret_cast<uint4 *>(row + (2 * i + 1) * 128) =
          make_uint4(e4m3x2_to_f16x2(w.z), e4m3x2_to_f16x2(w.z >> 16), e4m3x2_to_f16x2(w.w),
                     e4m3x2_to_f16x2(w.w >> 16));
    }
  }
}

__global__ void __launch_bounds__(kTcThreads, 2) attn_chunked_tc_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(1024) uint8_t s_dyn[];
  __shared__ __align__(8) uint64_t s_mbar[2];               // S done, P V done
  __shared__ uint32_t s_tmem;
  __shared__ float s_red[4][kTcMaxH];
  __shared__ float s_m[kTcMaxH], s_alpha[kTcMaxH];
  __shared__ int s_rescale;
  pdl_enter();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = tid & (kTcChunk - 1), half = tid >> 7;      // key row / TMEM lane / dim, and head-dim half
  const int H = a.H;                                         // <= kTcMaxH, a multiple of 16
  const int h_lo = 32 * half;                                // this thread's heads: h_lo .. h_lo + 31
  const bool heads = h_lo < H;
  uint8_t *qs = s_dyn + kTcQ, *ks = s_dyn + kTcK, *ps = s_dyn + kTcP, *ps2 = s_dyn + kTcP2;
  const uint32_t mb_s = smem_addr(&s_mbar[0]), mb_pv = smem_addr(&s_mbar[1]);

  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(mb_s));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(mb_pv));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (tid < 64) reinterpret_cast<__half *>(s_dyn + kTcOnes)[tid] = __float2half(1.f);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(&s_tmem)),
                 "r"(kTcCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t t_s = tmem, t_o = tmem + kTcMaxH, t_l = tmem + 2 * kTcMaxH;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;   // this warp's TMEM lanes
  const uint32_t id_s = umma_idesc(kTcChunk, H, 0, 0);       // S^T = K Q^T
  const uint32_t id_o = umma_idesc(kD, H, 1, 1);             // O^T += V^T P^T, l += 1 P^T
  uint32_t ph_s = 0, ph_pv = 0;
  bool pv_pending = false, dead = false;   // dead: a wait ran out (uniform across the CTA)
  const float ltau = a.tau * kTcLog2e;
  constexpr int kQPer = kTcMaxH * 16 / kTcThreads;           // 16-byte query chunks per thread

  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    // ---- every load the row start needs, issued together: the row's identity, its queries
    // and the first chunk's indices; then its sequence base and the first key rows
    const int b = a.q_seq[t];
    const int64_t p = a.q_pos[t];
    const int32_t idx0 = (a.n_sel_chunks > 0 && k < a.topk) ? __ldg(a.topk_idx + t * a.topk + k) : -1;
    uint4 qv[kQPer];
#pragma unroll
    for (int j = 0; j < kQPer; ++j) {
      const int i = tid + j * kTcThreads, h = i >> 4, dg = i & 15;
      qv[j] = h < H ? __ldg(reinterpret_cast<const uint4 *>(a.q + ((int64_t)t * H + h) * kD + 8 * dg))
                    : make_uint4(0, 0, 0, 0);
    }
    bool ok = b >= 0 && b < a.c.B;
    int64_t base = 0;
    if (ok) {
      base = a.c.seq_base[b];
      const int64_t len = a.c.seq_len[b];
      ok = p >= 0 && p < len && base >= 0 && base + len <= a.c.T_cap;
    }
    if (!ok && tid == 0) set_err(a.d_err, (b < 0 || b >= a.c.B) ? CSA2_DEVERR_SEQ : CSA2_DEVERR_POS);
    KeyRaw kr;
    {
      int64_t rp;
      key_slot(a, 0, k, t, idx0, true, p, kr, rp);
      if (!ok) kr.valid = false;
      key_fetch(a, half, b, base, rp, kr);
    }
    // the previous row's last products are complete: Q may be overwritten
#pragma unroll
    for (int j = 0; j < kQPer; ++j) {
      const int i = tid + j * kTcThreads, h = i >> 4, dg = i & 15;
      if (h < H) {
        const uint32_t w[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
        uint32_t o4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) o4[q] = pack_f16x2(bf16_to_f32(w[q] & 0xFFFFu), bf16_to_f32(w[q] >> 16));
        *reinterpret_cast<uint4 *>(qs + ((h >> 3) * 16 + dg) * 128 + (h & 7) * 16) =
            make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
    }
    if (tid < kTcMaxH) s_m[tid] = -INFINITY;

    for (int c = 0; c < a.n_chunks; ++c) {
      // ---- K and P are free once the previous P V product has completed
      bool waited = true;
      if (pv_pending) {
        waited = mbar_wait(mb_pv, ph_pv);
        ph_pv ^= 1u;
        pv_pending = false;
        tc_fence_after();
      }
      store_key(ks, k, half, kr);
      const bool fp8 = kr.fp8, valid = kr.valid;
      const float wsc = kr.wsc;
      if (c + 1 < a.n_chunks) {                              // the next chunk's rows
        int64_t rp;
        key_slot(a, c + 1, k, t, 0, false, p, kr, rp);
        if (!ok) kr.valid = false;
        key_fetch(a, half, b, base, rp, kr);
      }
      fence_async_smem();
      tc_fence_before();
      if (__syncthreads_or(!waited)) { dead = true; break; }   // a product never completed: stop
      tc_fence_after();
      if (tid == 0) {
#pragma unroll
        for (int s = 0; s < kD / 16; ++s)
          umma_f16(t_s, umma_desc(smem_addr(ks) + 256 * s, 128, 2048), umma_desc(smem_addr(qs) + 256 * s, 128, 2048),
                   id_s, s > 0);
        umma_commit(mb_s);
      }
      __syncwarp();
      const bool s_done = mbar_wait(mb_s, ph_s);
      ph_s ^= 1u;
      tc_fence_after();

      // ---- scores of this key row for this thread's heads; chunk maxima per head
      const float rs = fp8 ? ltau * wsc : ltau;                // log2-domain scale of this row's scores
      float sv[32];
      {
        float v[32];
        if (heads) tmem_ld32(t_s + lane_off + h_lo, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[j] = (heads && h_lo + j < H && valid) ? v[j] * rs : -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float m = warp_max_f32(sv[j]);
        if (lane == j) s_red[warp & 3][h_lo + j] = m;
      }
      if (__syncthreads_or(!s_done)) { dead = true; break; }
      if (tid < H) {
        const float m_old = s_m[tid];
        const float m_new = fmaxf(m_old, fmaxf(fmaxf(s_red[0][tid], s_red[1][tid]), fmaxf(s_red[2][tid], s_red[3][tid])));
        s_alpha[tid] = (m_old == -INFINITY || m_old == m_new) ? 1.f : exp2f(m_old - m_new);
        s_m[tid] = m_new;
      }
      if (tid == 0) s_rescale = 0;
      __syncthreads();
      if (tid < H && s_alpha[tid] != 1.f) s_rescale = 1;

      // ---- P^T row of this key (f16).  A window row's values are its E4M3 codes, so its
      // float32 scale multiplies P for O; the row sums take P without it (second copy).
      if (heads) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (h_lo + 8 * q < H) {
            float pr[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float x = sv[8 * q + j];
              pr[j] = x == -INFINITY ? 0.f : exp2f(x - s_m[h_lo + 8 * q + j]);
            }
            const int off = ((k >> 3) * (kTcMaxH / 8) + (h_lo >> 3) + q) * 128 + (k & 7) * 16;
            if (fp8) {
              *reinterpret_cast<uint4 *>(ps2 + off) = make_uint4(pack_f16x2(pr[0], pr[1]), pack_f16x2(pr[2], pr[3]),
                                                                 pack_f16x2(pr[4], pr[5]), pack_f16x2(pr[6], pr[7]));
#pragma unroll
              for (int j = 0; j < 8; ++j) pr[j] *= wsc;
            }
            *reinterpret_cast<uint4 *>(ps + off) = make_uint4(pack_f16x2(pr[0], pr[1]), pack_f16x2(pr[2], pr[3]),
                                                              pack_f16x2(pr[4], pr[5]), pack_f16x2(pr[6], pr[7]));
          }
        }
      }
      __syncthreads();
      // ---- a head's maximum grew: rescale its O^T column and its row sum
      if (c > 0 && s_rescale && heads) {
        float v[32], u[32];
        tmem_ld32(t_o + lane_off + h_lo, v);
        tmem_ld32(t_l + lane_off + h_lo, u);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float al = s_alpha[h_lo + j];
          v[j] *= al;
          u[j] *= al;
        }
        tmem_st32(t_o + lane_off + h_lo, v);
        tmem_st32(t_l + lane_off + h_lo, u);
        tmem_st_wait();
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {
        const uint32_t pl = smem_addr(c >= a.n_sel_chunks ? ps2 : ps);   // P for the row sums
#pragma unroll
        for (int s = 0; s < kTcChunk / 16; ++s) {
          const uint32_t koff = 2 * (kTcMaxH / 8) * 128 * s;
          const uint64_t bd = umma_desc(smem_addr(ps) + koff, (kTcMaxH / 8) * 128, 128);
          const uint64_t bl = umma_desc(pl + koff, (kTcMaxH / 8) * 128, 128);
          const uint32_t acc = (c > 0 || s > 0) ? 1u : 0u;
          umma_f16(t_o, umma_desc(smem_addr(ks) + 2 * 2048 * s, 2048, 128), bd, id_o, acc);
          umma_f16(t_l, umma_desc(smem_addr(s_dyn + kTcOnes), 0, 0), bl, id_o, acc);
        }
        umma_commit(mb_pv);
      }
      __syncwarp();
      pv_pending = true;
    }

    if (dead) break;
    // ---- O = O^T / l: thread (d, half) holds dim d of heads h_lo .. h_lo + 31
    bool waited = true;
    if (pv_pending) {
      waited = mbar_wait(mb_pv, ph_pv);
      ph_pv ^= 1u;
      pv_pending = false;
      tc_fence_after();
    }
    if (__syncthreads_or(!waited)) { dead = true; break; }
    const int64_t head0 = (int64_t)t * H;
    if (heads) {
      float v[32], u[32];
      tmem_ld32(t_o + lane_off + h_lo, v);
      tmem_ld32(t_l + lane_off + h_lo, u);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (h_lo + j < H) {
          const float l = u[j];                               // every lane holds every head's sum
          a.out[(head0 + h_lo + j) * kD + k] = l > 0.f ? v[j] / l : 0.f;
          if (a.lse && k == j)
            a.lse[head0 + h_lo + j] = l > 0.f ? s_m[h_lo + j] / kTcLog2e + logf(l) : -INFINITY;
        }
      }
    }
    tc_fence_before();
    __syncthreads();                                          // s_m and TMEM reads done before the next row
    tc_fence_after();
  }
  if (dead && tid == 0) set_err(a.d_err, CSA2_DEVERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTcCols));
}

// ------------------------------------------------------------------ host side

bool attn_tc_eligible(int64_t T, int H) { return H >= 16 && H <= kTcMaxH && (H % 16) == 0 && T * H >= 64 * 256; }

cudaError_t launch_attn_chunked_tc(const csa2_cache &c, const csa2_swa &swa, const uint16_t *q, int H, int64_t T,
                                   const int32_t *q_seq, const int64_t *q_pos, const int32_t *topk_idx, int topk,
                                   int window, float tau, float *out, float *lse, int32_t *d_err, cudaStream_t st) {
  opt_in_smem((const void *)attn_chunked_tc_kernel, kTcSmemLaunch, kSiteAttnTcOptin, 0);
  TcArgs a;
  a.c = c; a.swa = swa; a.q = q; a.H = H; a.T = T; a.q_seq = q_seq; a.q_pos = q_pos;
  a.topk_idx = topk_idx; a.topk = topk; a.window = window; a.tau = tau; a.out = out; a.lse = lse; a.d_err = d_err;
  a.n_sel_chunks = (topk + kTcChunk - 1) / kTcChunk;
  a.n_chunks = a.n_sel_chunks + (window + kTcChunk - 1) / kTcChunk;
  const int64_t grid = std::min<int64_t>(T, (int64_t)num_sms() * 2);
  return launch_k(attn_chunked_tc_kernel, dim3((unsigned)grid), dim3(kTcThreads), kTcSmemLaunch, st, 0, a);
}

}  // namespace csa2
