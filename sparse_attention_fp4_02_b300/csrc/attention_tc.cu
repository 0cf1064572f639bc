// Chunked-query sparse attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Method: as sparse_attn_decode (ttj.kr "DeepSeek-V4.1-Flash, KV 캐시를 토큰당 890바이트까지
// 압축하다", section "CSA2와 어텐션 재설계"; origotech.dev deep dive, subsection "Compressed
// Sparse Attention 2(CSA2)"): one softmax over a row's selected FP4 rows plus its FP8
// window, V = K.  With many query rows and 64 heads every gathered key row is shared by all
// heads of its query row, so the two products are dense contractions, per chunk of 128 keys:
//   S = Q K^T      (M = 64 heads, N = 128 keys, K = 128 dims)
//   O += P V       (M = 64 heads, N = 128 dims, K = 128 keys)
//
// One persistent CTA per SM walks its query rows as one stream of (row, chunk) steps, with
// three roles that hand stages to each other through mbarriers, so that the gathers, the
// tensor cores and the softmax of different chunks overlap:
//   * producer warps (4): thread k gathers key row k of a chunk with cp.async into a
//     4-deep ring of raw stages (the top-k index and the row's sequence entry are loaded a
//     step ahead), then dequantises it exactly into f16 core matrices of one of two K
//     stages (the same bytes serve as K, K-major, for S and, read MN-major, as V for O); at
//     a row's first chunk they also write its queries (bf16 -> f16) into one of two Q
//     stages;
//   * one MMA thread: S of step u into one of two TMEM S buffers as soon as its keys are
//     in, then O += P V of step u - 1 into the row's TMEM O buffer (two, by row parity)
//     once its P is written;
//   * softmax warps (4): an M = 64 accumulator puts head h in TMEM lane 32 (h / 16) + h %
//     16, so lanes 0-15 of warp w own heads 16 w .. 16 w + 15, each with all 128 scores of
//     a chunk in its own registers: chunk maximum, P = 2^(s - m) in f16 to shared memory,
//     the row sum in float32, and at a row's end O / l and the log-sum-exp.  The reference
//     maximum m is raised (and O rescaled in TMEM) only when a chunk's maximum exceeds it
//     by more than a factor 2^8, so P stays below 2^8 and the rescale is rare; the softmax
//     is the same for any common reference.
//
// Exactness of the operands: an E2M1 value times its E4M3 group scale has at most 6
// significant bits within [2^-10, 2688] and is exact in f16; an E4M3 value is exact in
// f16 (the window's float32 row scale multiplies its scores and its P instead).
#include <cfloat>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace csa2 {

constexpr int kTcChunk = 128;            // key rows per chunk (N of S, K of P V)
constexpr int kTcMaxH = 64;              // heads per row (M of both products)
constexpr int kWsThreads = 9 * 32;       // softmax warps 0-3, producer warps 4-7, MMA warp 8
constexpr int kWsRaw = 4;                // raw gather stages per producer thread
constexpr int kRawKey = 144;             // bytes of one key row in a raw stage: 128 codes + scales
constexpr float kTcLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.f;      // raise the reference maximum only past a factor 2^8

// dynamic shared memory (bytes); every operand is K-major (V: MN-major) in 8 x 16-byte core
// matrices, block (group of 8 rows, group of 8 K elements) at group * 2048 + kgroup * 128
constexpr int kQBytes = kTcMaxH * kD * 2;                 // 64 heads x 128 dims f16   16 KB
constexpr int kKBytes = kTcChunk * kD * 2;                // 128 keys x 128 dims f16   32 KB
constexpr int kPBytes = kTcMaxH * kTcChunk * 2;           // 64 heads x 128 keys f16   16 KB
constexpr int kRawStage = kTcChunk * kRawKey;             // 18 KB
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + 2 * kQBytes;
constexpr int kOffP = kOffK + 2 * kKBytes;
constexpr int kOffRaw = kOffP + 2 * kPBytes;
constexpr int kOffKf = kOffRaw + kWsRaw * kRawStage;      // [stage][kmul | kval][128] float
constexpr int kOffUni = kOffKf + 2 * 2 * kTcChunk * 4;    // [stage][4 producer warps] int
constexpr int kWsSmem = kOffUni + 2 * 4 * 4;
static_assert(kWsSmem <= 227 * 1024, "one CTA per SM");
constexpr int kWsCols = 512;             // TMEM columns: S buffers at 0 and 128, O buffers at 256 and 384

// mbarriers; the k-th completion of a stage-x barrier belongs to step (or row) x + 2k
enum {
  kBarKFull = 0,     // [2] keys of a step (and at a row's first step its queries) in: 4 producer-warp arrivals
  kBarSFull = 2,     // [2] S of a step in its TMEM buffer: MMA commit
  kBarPFull = 4,     // [2] P of a step written and O rescaled: 4 softmax-warp arrivals
  kBarPvDone = 6,    // [2] P V of a step complete: MMA commit
  kBarQEmpty = 8,    // [2] every S of a row complete (its Q stage is free): MMA commit
  kBarOEmpty = 10,   // [2] a row's O buffer read out: 4 softmax-warp arrivals
  kBarFin = 12,      // every MMA issued has completed
  kNumBars = 13
};

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

__device__ __forceinline__ uint32_t fp4x2_f16x2(uint32_t byte) {
  __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)(byte & 0xFFu), __NV_E2M1);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async4_raw(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src));
}
// bounded wait taken by a whole warp: every lane gets the same answer, so that no lane leaves
// the warp's collective steps alone
__device__ __forceinline__ bool mbar_wait_warp(uint32_t mbar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(mbar, parity));
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(mbar) : "memory");
}

// 32 consecutive TMEM columns of this thread's lane: the load, then a wait that every use of
// the registers depends on
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

__global__ void __launch_bounds__(kWsThreads, 1) attn_chunked_tc_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(16) uint8_t s_dyn[];
  __shared__ __align__(8) uint64_t s_bar[kNumBars];
  __shared__ uint32_t s_tmem;
  pdl_enter();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t G = gridDim.x;
  const int64_t nrows = a.T > (int64_t)blockIdx.x ? (a.T - 1 - (int64_t)blockIdx.x) / G + 1 : 0;
  const int NC = a.n_chunks;
  const int64_t U = nrows * NC;                              // (row, chunk) steps of this CTA
  auto bar = [&](int i) { return smem_addr(&s_bar[i]); };

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const int cnt = (i < kBarSFull || (i >= kBarPFull && i < kBarPvDone) || (i >= kBarOEmpty && i < kBarFin)) ? 4 : 1;
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar(i)), "r"(cnt));
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(&s_tmem)),
                 "r"(kWsCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  // queries of heads >= H stay zero in both Q stages (their rows of S and O are never read)
  for (int i = tid; i < 2 * kQBytes / 16; i += kWsThreads)
    reinterpret_cast<uint4 *>(s_dyn + kOffQ)[i] = make_uint4(0, 0, 0, 0);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool dead = false;                                         // a bounded wait gave up: leave the loop

  if (warp == 8) {
    // ================================================================ MMA issue (one thread)
    if (lane == 0 && U > 0) {
      const uint32_t id_s = umma_idesc(kTcMaxH, kTcChunk, 0, 0);   // S = Q K^T: A, B K-major
      const uint32_t id_o = umma_idesc(kTcMaxH, kD, 0, 1);         // O += P V: A K-major, B MN-major
      const uint32_t q_a = smem_addr(s_dyn + kOffQ), k_a = smem_addr(s_dyn + kOffK), p_a = smem_addr(s_dyn + kOffP);
      const uint64_t dq0 = umma_desc(q_a, 128, 2048), dq1 = umma_desc(q_a + kQBytes, 128, 2048);
      const uint64_t dk0 = umma_desc(k_a, 128, 2048), dk1 = umma_desc(k_a + kKBytes, 128, 2048);
      const uint64_t dv0 = umma_desc(k_a, 2048, 128), dv1 = umma_desc(k_a + kKBytes, 2048, 128);
      const uint64_t dp0 = umma_desc(p_a, 128, 2048), dp1 = umma_desc(p_a + kPBytes, 128, 2048);
      // P V of step v (row iv, chunk cv); the descriptors advance 16 keys per MMA
      auto issue_pv = [&](int64_t v, int64_t iv, int cv) -> bool {
        const int x = (int)(v & 1);
        if (cv == 0 && iv >= 2 && !mbar_wait(bar(kBarOEmpty + (int)(iv & 1)), (uint32_t)(((iv - 2) >> 1) & 1)))
          return false;
        if (!mbar_wait(bar(kBarPFull + x), (uint32_t)((v >> 1) & 1))) return false;
        tc_fence_after();
        const uint32_t d = tmem + 256 + 128 * (uint32_t)(iv & 1);
        const uint64_t dp = x ? dp1 : dp0, dv = x ? dv1 : dv0;
#pragma unroll
        for (int s = 0; s < kTcChunk / 16; ++s)
          umma_f16(d, dp + (uint64_t)(16 * s), dv + (uint64_t)(256 * s), id_o, (cv > 0 || s > 0) ? 1u : 0u);
        umma_commit(bar(kBarPvDone + x));
        return true;
      };
      int64_t i = 0, pi = 0;
      int c = 0, pc = 0;                                     // (row, chunk) of step u and of step u - 1
      for (int64_t u = 0; u < U; ++u) {
        const int x = (int)(u & 1);
        if (!mbar_wait(bar(kBarKFull + x), (uint32_t)((u >> 1) & 1))) { dead = true; break; }
        tc_fence_after();
        const uint64_t dq = (i & 1) ? dq1 : dq0, dk = x ? dk1 : dk0;
#pragma unroll
        for (int s = 0; s < kD / 16; ++s)
          umma_f16(tmem + 128 * (uint32_t)x, dq + (uint64_t)(16 * s), dk + (uint64_t)(16 * s), id_s, s > 0 ? 1u : 0u);
        umma_commit(bar(kBarSFull + x));
        if (c == NC - 1) umma_commit(bar(kBarQEmpty + (int)(i & 1)));
        if (u >= 1 && !issue_pv(u - 1, pi, pc)) { dead = true; break; }
        pi = i;
        pc = c;
        if (++c == NC) { c = 0; ++i; }
      }
      if (!dead) dead = !issue_pv(U - 1, pi, pc);
      // every MMA issued has completed before TMEM is released
      umma_commit(bar(kBarFin));
      if (!mbar_wait(bar(kBarFin), 0)) dead = true;
    }
  } else if (warp >= 4) {
    // ================================================================ producers
    const int pt = tid - 128, pw = pt >> 5;                  // key row pt of every chunk
    const uint32_t raw_s = smem_addr(s_dyn + kOffRaw + pt * kRawKey);
    const uint8_t *raw_g = s_dyn + kOffRaw + pt * kRawKey;
    float *kf = reinterpret_cast<float *>(s_dyn + kOffKf);
    int *kuni = reinterpret_cast<int *>(s_dyn + kOffUni);
    const int krow = (pt >> 3) * 2048 + (pt & 7) * 16;      // this key's core-matrix rows
    const float ltau = a.tau * kTcLog2e;
    const int nsel = a.n_sel_chunks;
    auto row_t = [&](int64_t i) -> int64_t { return (int64_t)blockIdx.x + i * G; };

    // row entries, loaded ahead so that no load waits on another at a row start:
    // (b, p) two rows ahead of the issue cursor, (base, len) one row ahead
    int nb1 = -1, nb2 = -1;
    int64_t np1 = 0, np2 = 0, nbase1 = 0, nlen1 = 0;
    if (nrows > 0) { nb1 = a.q_seq[row_t(0)]; np1 = a.q_pos[row_t(0)]; }
    if (nrows > 1) { nb2 = a.q_seq[row_t(1)]; np2 = a.q_pos[row_t(1)]; }
    if (nb1 >= 0 && nb1 < a.c.B) { nbase1 = a.c.seq_base[nb1]; nlen1 = a.c.seq_len[nb1]; }
    int cb = 0;                                              // the issue cursor's row entry
    int64_t cp = 0, cbase = 0;
    bool cok = false;
    int64_t ii = 0;                                          // the issue cursor (row, chunk)
    int ic = 0;
    auto load_idx = [&](int64_t i, int c) -> int32_t {
      if (i >= nrows || c >= nsel) return -1;
      const int j = c * kTcChunk + pt;
      return j < a.topk ? __ldg(a.topk_idx + row_t(i) * a.topk + j) : -1;
    };
    int32_t idx_next = load_idx(0, 0);                       // top-k index of the next issued step
    uint32_t vbits = 0, fbits = 0;                           // per raw stage: valid row, FP8 row
    auto issue = [&](int64_t v) {
      const int slot = (int)(v % kWsRaw);
      if (v < U) {
        if (ic == 0) {                                       // entering row ii: rotate the entries
          cb = nb1;
          cp = np1;
          cbase = nbase1;
          const int64_t clen = nlen1;
          cok = cb >= 0 && cb < a.c.B;
          if (cok) cok = cp >= 0 && cp < clen && cbase >= 0 && cbase + clen <= a.c.T_cap;
          if (!cok && pt == 0) set_err(a.d_err, (cb < 0 || cb >= a.c.B) ? CSA2_DEVERR_SEQ : CSA2_DEVERR_POS);
          nb1 = nb2;
          np1 = np2;
          nbase1 = 0;
          nlen1 = 0;
          if (ii + 1 < nrows && nb1 >= 0 && nb1 < a.c.B) { nbase1 = a.c.seq_base[nb1]; nlen1 = a.c.seq_len[nb1]; }
          nb2 = -1;
          np2 = 0;
          if (ii + 2 < nrows) { nb2 = a.q_seq[row_t(ii + 2)]; np2 = a.q_pos[row_t(ii + 2)]; }
        }
        const uint32_t dst = raw_s + slot * kRawStage;
        const bool fp8 = ic >= nsel;
        bool valid;
        if (!fp8) {
          const int32_t idx = idx_next;
          if (cok && idx >= 0 && idx > cp) set_err(a.d_err, CSA2_DEVERR_INDEX);
          valid = cok && idx >= 0 && idx <= cp;
          if (valid) {
            const int64_t row = cbase + idx;
            const uint8_t *src = a.c.kv_codes + row * (kD / 2);
#pragma unroll
            for (int q = 0; q < 4; ++q) cp_async16(dst + 16 * q, src + 16 * q, true);
            cp_async8(dst + 128, a.c.kv_scales + row * (kD / 16));
          }
        } else {
          const int j = (ic - nsel) * kTcChunk + pt;
          const int64_t pj = cp - a.window + 1 + j;
          valid = cok && j < a.window && pj >= 0;
          if (valid) {
            const int64_t srow = (int64_t)cb * a.swa.ring + pj % a.swa.ring;
            const uint8_t *src = a.swa.codes + srow * kD;
#pragma unroll
            for (int q = 0; q < 8; ++q) cp_async16(dst + 16 * q, src + 16 * q, true);
            cp_async4_raw(dst + 128, a.swa.scale + srow);
          }
        }
        vbits = (vbits & ~(1u << slot)) | ((valid ? 1u : 0u) << slot);
        fbits = (fbits & ~(1u << slot)) | ((fp8 ? 1u : 0u) << slot);
        if (++ic == NC) { ic = 0; ++ii; }
        idx_next = load_idx(ii, ic);
      }
      cp_async_commit();
    };

    // queries of the next row to enter, in registers: piece pt + 128 j = (head, 8-dim group)
    uint4 qv[8];
    auto load_q = [&](int64_t i) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int pc = pt + 128 * j, h = pc >> 4, dg = pc & 15;
        qv[j] = (i < nrows && h < a.H)
                    ? __ldg(reinterpret_cast<const uint4 *>(a.q + (row_t(i) * a.H + h) * kD + 8 * dg))
                    : make_uint4(0, 0, 0, 0);
      }
    };
    load_q(0);
    for (int s = 0; s < kWsRaw; ++s) issue(s);

    int64_t i = 0;
    int c = 0;
    for (int64_t u = 0; u < U; ++u) {
      const int x = (int)(u & 1), slot = (int)(u % kWsRaw);
      cp_async_wait<kWsRaw - 1>();                           // this thread's copies of step u
      if (c == 0) {
        // the row's queries into Q stage i & 1, once every S of row i - 2 is complete
        if (i >= 2 && !mbar_wait_warp(bar(kBarQEmpty + (int)(i & 1)), (uint32_t)(((i - 2) >> 1) & 1))) { dead = true; break; }
        uint8_t *qs = s_dyn + kOffQ + (i & 1) * kQBytes;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int pc = pt + 128 * j, h = pc >> 4, dg = pc & 15;
          if (h < a.H) {
            const uint32_t w[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
            uint32_t o4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o4[e] = pack_f16x2(bf16_to_f32(w[e] & 0xFFFFu), bf16_to_f32(w[e] >> 16));
            *reinterpret_cast<uint4 *>(qs + ((h >> 3) * 16 + dg) * 128 + (h & 7) * 16) =
                make_uint4(o4[0], o4[1], o4[2], o4[3]);
          }
        }
        load_q(i + 1);
      }
      // K stage x is free once the P V of step u - 2 is complete
      if (u >= 2 && !mbar_wait_warp(bar(kBarPvDone + x), (uint32_t)(((u - 2) >> 1) & 1))) { dead = true; break; }
      const bool valid = (vbits >> slot) & 1u, fp8 = (fbits >> slot) & 1u;
      uint8_t *kt = s_dyn + kOffK + x * kKBytes + krow;
      const uint8_t *raw = raw_g + slot * kRawStage;
      float kmul = 0.f, kval = -1.f;
      if (!valid) {
#pragma unroll
        for (int dg = 0; dg < 16; ++dg) *reinterpret_cast<uint4 *>(kt + dg * 128) = make_uint4(0, 0, 0, 0);
      } else if (!fp8) {
        const uint2 sc = *reinterpret_cast<const uint2 *>(raw + 128);
#pragma unroll
        for (int g = 0; g < 8; ++g) {                        // channels 16 g .. 16 g + 15: two core-matrix rows
          const uint32_t s16 = e4m3x2_to_f16x2(((g < 4 ? sc.x : sc.y) >> (8 * (g & 3))) & 0xFFu) & 0xFFFFu;
          const uint32_t s2 = s16 | (s16 << 16);
          const uint2 cw = *reinterpret_cast<const uint2 *>(raw + 8 * g);
          uint32_t v[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = hmul2_bits(fp4x2_f16x2(cw.x >> (8 * e)), s2);
#pragma unroll
          for (int e = 0; e < 4; ++e) v[4 + e] = hmul2_bits(fp4x2_f16x2(cw.y >> (8 * e)), s2);
          *reinterpret_cast<uint4 *>(kt + (2 * g) * 128) = make_uint4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<uint4 *>(kt + (2 * g + 1) * 128) = make_uint4(v[4], v[5], v[6], v[7]);
        }
        kmul = ltau;
        kval = 1.f;
      } else {
        const float wsc = *reinterpret_cast<const float *>(raw + 128);
#pragma unroll
        for (int g = 0; g < 8; ++g) {                        // codes 16 g .. 16 g + 15: two core-matrix rows
          const uint4 w = *reinterpret_cast<const uint4 *>(raw + 16 * g);
          *reinterpret_cast<uint4 *>(kt + (2 * g) * 128) = make_uint4(
              e4m3x2_to_f16x2(w.x), e4m3x2_to_f16x2(w.x >> 16), e4m3x2_to_f16x2(w.y), e4m3x2_to_f16x2(w.y >> 16));
          *reinterpret_cast<uint4 *>(kt + (2 * g + 1) * 128) = make_uint4(
              e4m3x2_to_f16x2(w.z), e4m3x2_to_f16x2(w.z >> 16), e4m3x2_to_f16x2(w.w), e4m3x2_to_f16x2(w.w >> 16));
        }
        kmul = ltau * wsc;
        kval = wsc;
      }
      kf[x * 2 * kTcChunk + pt] = kmul;
      kf[x * 2 * kTcChunk + kTcChunk + pt] = kval;
      const bool uni = __all_sync(0xffffffffu, valid && !fp8);
      if (lane == 0) kuni[x * 4 + pw] = uni ? 1 : 0;
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarKFull + x));
      issue(u + kWsRaw);                                     // the raw stage is free again
      if (++c == NC) { c = 0; ++i; }
    }
    cp_async_wait<0>();
  } else {
    // ================================================================ softmax (warps 0-3)
    const int h = 16 * warp + lane;                          // head of lanes 0-15
    const bool own = lane < 16 && h < a.H;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const float *kf = reinterpret_cast<const float *>(s_dyn + kOffKf);
    const int *kuni = reinterpret_cast<const int *>(s_dyn + kOffUni);
    const float ltau = a.tau * kTcLog2e;
    float m = -INFINITY, l = 0.f;
    int64_t i = 0;
    int c = 0;
    for (int64_t u = 0; u < U; ++u) {
      const int x = (int)(u & 1);
      const uint32_t par = (uint32_t)((u >> 1) & 1);
      if (!mbar_wait_warp(bar(kBarKFull + x), par) || !mbar_wait_warp(bar(kBarSFull + x), par)) { dead = true; break; }
      tc_fence_after();
      float s[kTcChunk];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        const uint32_t ts = tmem + lane_base + 128 * (uint32_t)x;
        tmem_ld32_issue(ts, r0);
        tmem_ld32_issue(ts + 32, r1);
        tmem_ld32_issue(ts + 64, r2);
        tmem_ld32_issue(ts + 96, r3);
        tmem_ld32_wait(r0);
        tmem_ld32_wait(r1);
        tmem_ld32_wait(r2);
        tmem_ld32_wait(r3);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          s[j] = __uint_as_float(r0[j]);
          s[32 + j] = __uint_as_float(r1[j]);
          s[64 + j] = __uint_as_float(r2[j]);
          s[96 + j] = __uint_as_float(r3[j]);
        }
      }
      const int4 un = *reinterpret_cast<const int4 *>(kuni + 4 * x);
      const bool uni = un.x && un.y && un.z && un.w;         // every key a valid top-k row
      const float *km = kf + x * 2 * kTcChunk, *kv = km + kTcChunk;
      // the chunk maximum over eight independent partial maxima (short dependency chains)
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
      if (uni) {
#pragma unroll
        for (int j = 0; j < kTcChunk; ++j) {
          s[j] *= ltau;
          mx[j & 7] = fmaxf(mx[j & 7], s[j]);
        }
      } else {
#pragma unroll
        for (int j4 = 0; j4 < kTcChunk / 4; ++j4) {
          const float4 f = *reinterpret_cast<const float4 *>(km + 4 * j4);
          const float4 g = *reinterpret_cast<const float4 *>(kv + 4 * j4);
          s[4 * j4 + 0] = g.x >= 0.f ? s[4 * j4 + 0] * f.x : -INFINITY;
          s[4 * j4 + 1] = g.y >= 0.f ? s[4 * j4 + 1] * f.y : -INFINITY;
          s[4 * j4 + 2] = g.z >= 0.f ? s[4 * j4 + 2] * f.z : -INFINITY;
          s[4 * j4 + 3] = g.w >= 0.f ? s[4 * j4 + 3] * f.w : -INFINITY;
#pragma unroll
          for (int e = 0; e < 4; ++e) mx[(4 * j4 + e) & 7] = fmaxf(mx[(4 * j4 + e) & 7], s[4 * j4 + e]);
        }
      }
      const float cmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // the reference maximum: the chunk's at a row's start, later raised past 2^8 only
      bool resc = false;
      float alpha = 1.f;
      if (c == 0) {
        m = cmax;
        l = 0.f;
      } else if (cmax > m + kRescaleLog2 || (m == -INFINITY && cmax > -INFINITY)) {
        resc = true;
        alpha = m == -INFINITY ? 0.f : ex2_approx(m - cmax);
        m = cmax;
      }
      // P stage x is free once the P V of step u - 2 is complete
      if (u >= 2 && !mbar_wait_warp(bar(kBarPvDone + x), (uint32_t)(((u - 2) >> 1) & 1))) { dead = true; break; }
      // P of this head's keys (f16, times the window rows' scales) into the A operand; the
      // row sum adds the unrounded values
      uint8_t *ps = s_dyn + kOffP + x * kPBytes + ((h >> 3) & 7) * 2048 + (h & 7) * 16;
      float lsp[4] = {0.f, 0.f, 0.f, 0.f};                  // four partial row sums
      if (uni) {
#pragma unroll
        for (int kg = 0; kg < kTcChunk / 8; ++kg) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float p0 = ex2_approx(s[8 * kg + 2 * e] - m), p1 = ex2_approx(s[8 * kg + 2 * e + 1] - m);
            lsp[e] += p0 + p1;
            w4[e] = pack_f16x2(p0, p1);
          }
          if (lane < 16) *reinterpret_cast<uint4 *>(ps + kg * 128) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      } else {
#pragma unroll
        for (int kg = 0; kg < kTcChunk / 8; ++kg) {
          const float4 g0 = *reinterpret_cast<const float4 *>(kv + 8 * kg);
          const float4 g1 = *reinterpret_cast<const float4 *>(kv + 8 * kg + 4);
          const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float z0 = s[8 * kg + 2 * e], z1 = s[8 * kg + 2 * e + 1];
            const float p0 = z0 == -INFINITY ? 0.f : ex2_approx(z0 - m);
            const float p1 = z1 == -INFINITY ? 0.f : ex2_approx(z1 - m);
            lsp[e] += p0 + p1;
            w4[e] = pack_f16x2(p0 * fmaxf(g[2 * e], 0.f), p1 * fmaxf(g[2 * e + 1], 0.f));
          }
          if (lane < 16) *reinterpret_cast<uint4 *>(ps + kg * 128) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      l = l * alpha + ((lsp[0] + lsp[1]) + (lsp[2] + lsp[3]));
      // a head's reference maximum rose: rescale its O row once the P V of step u - 1 is in
      // (the TMEM access is warp-wide, so the warp rescales when any of its heads needs it)
      if (__any_sync(0xffffffffu, own && resc)) {
        if (!mbar_wait_warp(bar(kBarPvDone + (x ^ 1)), (uint32_t)(((u - 1) >> 1) & 1))) { dead = true; break; }
        tc_fence_after();
        const uint32_t t_o = tmem + lane_base + 256 + 128 * (uint32_t)(i & 1);
        const float f = (own && resc) ? alpha : 1.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t r[32];
          tmem_ld32_issue(t_o + 32 * q, r);
          tmem_ld32_wait(r);
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * f;
          tmem_st32(t_o + 32 * q, v);
        }
        tmem_st_wait();
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + x));
      if (c == NC - 1) {
        // ---- the row's end: O / l and the log-sum-exp, then its O buffer is free
        if (!mbar_wait_warp(bar(kBarPvDone + x), par)) { dead = true; break; }
        tc_fence_after();
        const int64_t t = (int64_t)blockIdx.x + i * G;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const uint32_t t_o = tmem + lane_base + 256 + 128 * (uint32_t)(i & 1);
        float *orow = a.out + (t * a.H + (own ? h : 0)) * kD;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t r[32];
          tmem_ld32_issue(t_o + 32 * q, r);
          tmem_ld32_wait(r);
          if (own) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4 *>(orow + 32 * q + j) =
                  make_float4(__uint_as_float(r[j]) * inv, __uint_as_float(r[j + 1]) * inv,
                              __uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv);
          }
        }
        if (own && a.lse) a.lse[t * a.H + h] = l > 0.f ? m / kTcLog2e + logf(l) : -INFINITY;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarOEmpty + (int)(i & 1)));
      }
      if (++c == NC) { c = 0; ++i; }
    }
  }
  if (dead) set_err(a.d_err, CSA2_DEVERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kWsCols));
}

// ------------------------------------------------------------------ host side

bool attn_tc_eligible(int64_t T, int H) { return H >= 16 && H <= kTcMaxH && (H % 16) == 0 && T * H >= 64 * 256; }

cudaError_t launch_attn_chunked_tc(const csa2_cache &c, const csa2_swa &swa, const uint16_t *q, int H, int64_t T,
                                   const int32_t *q_seq, const int64_t *q_pos, const int32_t *topk_idx, int topk,
                                   int window, float tau, float *out, float *lse, int32_t *d_err, cudaStream_t st) {
  opt_in_smem((const void *)attn_chunked_tc_kernel, kWsSmem, kSiteAttnTcOptin, 0);
  TcArgs a;
  a.c = c; a.swa = swa; a.q = q; a.H = H; a.T = T; a.q_seq = q_seq; a.q_pos = q_pos;
  a.topk_idx = topk_idx; a.topk = topk; a.window = window; a.tau = tau; a.out = out; a.lse = lse; a.d_err = d_err;
  a.n_sel_chunks = (topk + kTcChunk - 1) / kTcChunk;
  a.n_chunks = a.n_sel_chunks + (window + kTcChunk - 1) / kTcChunk;
  const int64_t grid = std::min<int64_t>(T, (int64_t)num_sms());
  return launch_k(attn_chunked_tc_kernel, dim3((unsigned)grid), dim3(kWsThreads), kWsSmem, st, 0, a);
}

}  // namespace csa2
