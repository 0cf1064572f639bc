// Chunked-query sparse attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Method: as sparse_attn_decode (ttj.kr "DeepSeek-V4.1-Flash, KV 캐시를 토큰당 890바이트까지
// 압축하다", section "CSA2와 어텐션 재설계"; origotech.dev deep dive, subsection "Compressed
// Sparse Attention 2(CSA2)"): one softmax over a row's selected FP4 rows plus its FP8
// window, V = K.  With many query rows and 64 heads every gathered key row is shared by all
// heads of its query row, so the two products are dense contractions, per chunk of 128 keys:
//   S = Q K^T      (M = 64 heads, N = 128 keys, K = 128 dims)
//   O += P V       (M = 64 heads, N = 128 dims, K = 128 keys)
// One CTA (8 warps) owns one query row at a time: threads k and k + 128 dequantise the two
// halves of key row k of the chunk exactly into f16 core matrices in shared memory (the
// same bytes serve as K, K-major, for S and, read MN-major, as V for O), one thread issues
// the MMAs, and both accumulators live in TMEM.  An M = 64 accumulator puts head h in TMEM
// lane 32 (h / 16) + h % 16, so lanes 0-15 of each warp hold 16 heads' rows: each head's
// softmax is thread-local, shared by two threads (warps w and w + 4), one per half of the
// chunk's keys and one per half of the output dims.  The softmax is online across chunks:
// a head's running maximum, its rescaling of O in TMEM and its row sum (the same
// f16-rounded P the product uses, added in float32) all stay with the head's threads.
//
#include <cfloat>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace csa2 {

constexpr int kTcThreads = 256;          // 8 warps: threads k and k + 128 dequantise key row k
constexpr int kTcChunk = 128;            // key rows per chunk (N of S, K of P V)
constexpr int kTcMaxH = 64;              // heads per row (M of both products)
constexpr int kTcCols = 256;             // TMEM columns per CTA: S (128 keys) | O (128 dims)
constexpr float kTcLog2e = 1.4426950408889634f;

// dynamic shared memory layout (bytes); every operand is K-major (V: MN-major) in 8 x 16-byte
// core matrices, block (group of 8 rows, group of 8 K elements) at group * 2048 + kgroup * 128
constexpr int kTcQ = 0;                                   // Q: 64 heads x 128 dims f16         16 KB
constexpr int kTcK = kTcQ + kTcMaxH * kD * 2;             // K chunk: 128 keys x 128 dims f16   32 KB
constexpr int kTcP = kTcK + kTcChunk * kD * 2;            // P: 64 heads x 128 keys f16         16 KB
constexpr int kTcSmem = kTcP + kTcMaxH * kTcChunk * 2;
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
  __shared__ __align__(16) float s_kmul[kTcChunk];          // per key of the chunk: score factor (log2 domain)
  __shared__ __align__(16) float s_kval[kTcChunk];          //   and value factor (< 0: not a valid key)
  __shared__ float s_cmax[2][kTcMaxH];                      // chunk maxima of the two key halves
  __shared__ float s_lsum[2][kTcMaxH];                      // row sums of the two key halves
  pdl_enter();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = tid & (kTcChunk - 1), half = tid >> 7;      // dequantiser role: key row k, dims half
  const int H = a.H;                                         // <= kTcMaxH, a multiple of 16
  // softmax role (lanes 0-15): head m, keys / output dims half kh
  const int kh = warp >> 2, m = 16 * (warp & 3) + lane;
  const bool own = lane < 16 && m < H;
  uint8_t *qs = s_dyn + kTcQ, *ks = s_dyn + kTcK, *ps = s_dyn + kTcP;
  const uint32_t mb_s = smem_addr(&s_mbar[0]), mb_pv = smem_addr(&s_mbar[1]);

  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(mb_s));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(mb_pv));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(&s_tmem)),
                 "r"(kTcCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  // queries of heads >= H stay zero (their rows of S and O are never read)
  for (int i = tid; i < kTcMaxH * kD * 2 / 16; i += kTcThreads) reinterpret_cast<uint4 *>(qs)[i] = make_uint4(0, 0, 0, 0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;   // this warp's TMEM lanes
  const uint32_t t_s = tmem + lane_base + 64 * kh;                // this thread's 64 keys of S
  const uint32_t t_o = tmem + lane_base + kTcChunk + 64 * kh;     // this thread's 64 dims of O
  const uint32_t id_s = umma_idesc(kTcMaxH, kTcChunk, 0, 0);      // S = Q K^T: A, B K-major
  const uint32_t id_o = umma_idesc(kTcMaxH, kD, 0, 1);            // O += P V: A K-major, B MN-major
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
    float run_m = -INFINITY, lsum = 0.f;                     // this head's running maximum and row sum

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
      if (half == 0) {
        s_kmul[k] = kr.valid ? (kr.fp8 ? ltau * kr.wsc : ltau) : 0.f;
        s_kval[k] = kr.valid ? (kr.fp8 ? kr.wsc : 1.f) : -1.f;
      }
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
          umma_f16(tmem, umma_desc(smem_addr(qs) + 256 * s, 128, 2048), umma_desc(smem_addr(ks) + 256 * s, 128, 2048),
                   id_s, s > 0);
        umma_commit(mb_s);
      }
      __syncwarp();
      const bool s_done = mbar_wait(mb_s, ph_s);
      ph_s ^= 1u;
      tc_fence_after();

      // ---- this head's scores of its 64 keys (log2 domain); the chunk maximum
      float sv[64];
      {
        float v[32];
        tmem_ld32(t_s, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[j] = v[j];
        tmem_ld32(t_s + 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[32 + j] = v[j];
      }
      float cm = -INFINITY;
#pragma unroll
      for (int j4 = 0; j4 < 16; ++j4) {
        const float4 km = *reinterpret_cast<const float4 *>(&s_kmul[64 * kh + 4 * j4]);
        const float4 kv = *reinterpret_cast<const float4 *>(&s_kval[64 * kh + 4 * j4]);
        sv[4 * j4 + 0] = kv.x >= 0.f ? sv[4 * j4 + 0] * km.x : -INFINITY;
        sv[4 * j4 + 1] = kv.y >= 0.f ? sv[4 * j4 + 1] * km.y : -INFINITY;
        sv[4 * j4 + 2] = kv.z >= 0.f ? sv[4 * j4 + 2] * km.z : -INFINITY;
        sv[4 * j4 + 3] = kv.w >= 0.f ? sv[4 * j4 + 3] * km.w : -INFINITY;
        cm = fmaxf(cm, fmaxf(fmaxf(sv[4 * j4], sv[4 * j4 + 1]), fmaxf(sv[4 * j4 + 2], sv[4 * j4 + 3])));
      }
      if (lane < 16) s_cmax[kh][m] = cm;
      if (__syncthreads_or(!s_done)) { dead = true; break; }
      const float m_new = fmaxf(run_m, fmaxf(s_cmax[0][m & (kTcMaxH - 1)], s_cmax[1][m & (kTcMaxH - 1)]));
      const float alpha = (run_m == -INFINITY || run_m == m_new) ? 1.f : exp2f(run_m - m_new);
      run_m = m_new;

      // ---- P (f16) of this head's keys into the A operand; the row sum adds the same f16 P
      // (a window row's float32 scale multiplies P for O only)
      if (own) {
        float ls = 0.f;
#pragma unroll
        for (int g = 0; g < 8; ++g) {                          // keys 64 kh + 8 g .. + 7
          uint32_t w4[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int i0 = 8 * g + 2 * j;
            const float p0 = sv[i0] == -INFINITY ? 0.f : exp2f(sv[i0] - m_new);
            const float p1 = sv[i0 + 1] == -INFINITY ? 0.f : exp2f(sv[i0 + 1] - m_new);
            const __half2 h2 = __floats2half2_rn(p0, p1);
            const float2 f2 = __half22float2(h2);
            ls += f2.x + f2.y;
            const float v0 = s_kval[64 * kh + i0], v1 = s_kval[64 * kh + i0 + 1];
            w4[j] = (v0 == 1.f && v1 == 1.f) ? *reinterpret_cast<const uint32_t *>(&h2)
                                             : pack_f16x2(p0 * fmaxf(v0, 0.f), p1 * fmaxf(v1, 0.f));
          }
          const int kg = 8 * kh + g;                           // key group of the chunk
          *reinterpret_cast<uint4 *>(ps + ((m >> 3) * 16 + kg) * 128 + (m & 7) * 16) =
              make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        lsum = lsum * alpha + ls;
      }
      // ---- a head's maximum grew: rescale its O row (this thread's 64 dims); the TMEM
      // access is warp-wide, so the warp rescales when any of its heads needs it
      if (c > 0 && __any_sync(0xffffffffu, own && alpha != 1.f)) {
        float v[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          tmem_ld32(t_o + 32 * hh, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= alpha;
          tmem_st32(t_o + 32 * hh, v);
        }
        tmem_st_wait();
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {
#pragma unroll
        for (int s = 0; s < kTcChunk / 16; ++s)
          umma_f16(tmem + kTcChunk, umma_desc(smem_addr(ps) + 256 * s, 128, 2048),
                   umma_desc(smem_addr(ks) + 2 * 2048 * s, 2048, 128), id_o, (c > 0 || s > 0) ? 1u : 0u);
        umma_commit(mb_pv);
      }
      __syncwarp();
      pv_pending = true;
    }

    if (dead) break;
    // ---- O / l: thread (m, kh) writes dims 64 kh .. 64 kh + 63 of head m
    bool waited = true;
    if (pv_pending) {
      waited = mbar_wait(mb_pv, ph_pv);
      ph_pv ^= 1u;
      pv_pending = false;
      tc_fence_after();
    }
    if (lane < 16) s_lsum[kh][m] = lsum;
    if (__syncthreads_or(!waited)) { dead = true; break; }
    const float l = s_lsum[0][m & (kTcMaxH - 1)] + s_lsum[1][m & (kTcMaxH - 1)];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float *orow = a.out + ((int64_t)t * H + m) * kD + 64 * kh;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float v[32];
      tmem_ld32(t_o + 32 * hh, v);
      if (own) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4 *>(orow + 32 * hh + j) =
              make_float4(v[j] * inv, v[j + 1] * inv, v[j + 2] * inv, v[j + 3] * inv);
      }
    }
    if (own && kh == 0 && a.lse) a.lse[(int64_t)t * H + m] = l > 0.f ? run_m / kTcLog2e + logf(l) : -INFINITY;
    tc_fence_before();
    __syncthreads();                                          // TMEM reads and s_lsum done before the next row
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
