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
// tensor cores and the softmax of different steps overlap:
//   * producer warps (4): thread k gathers key row k of a step with cp.async into a 3-deep
//     ring of raw stages (the top-k index and the row's sequence entry are loaded a step
//     ahead), then dequantises it exactly into f16 core matrices of one of three K stages
//     (the same bytes serve as K, K-major, for S and, read MN-major, as V for O); at a
//     row's first step they also write its queries (bf16 -> f16) into one of two Q stages;
//   * one MMA thread: S of step u into one of two TMEM S buffers as soon as its keys are
//     in, then O += P V of step u - 1 into the row's TMEM O buffer (two, by row parity)
//     once its P is written;
//   * softmax warps (8): an M = 64 accumulator puts head h in TMEM lane 32 (h / 16) + h %
//     16; two warps share each lane quarter, one per half of the step's keys (and of the
//     output dims), and the 16x256b TMEM load gives thread t heads 16 q + t / 4 and
//     16 q + 8 + t / 4 with the key pairs 8 j + 2 (t % 4), + 1 of its half, so every lane
//     works.  Per head: the step's maximum (over a quad, then over the partner warp through
//     shared memory), P = 2^(s - m) in f16 to shared memory, the row sum in float32, and at
//     a row's end O / l and the log-sum-exp.  The reference maximum m is raised (and O
//     rescaled in TMEM) only when a step's maximum exceeds it by more than a factor 2^8, so
//     P stays below 2^8 and the rescale is rare; the softmax is the same for any common
//     reference.
//
// Exactness of the operands: an E2M1 value times its E4M3 group scale has at most 6
// significant bits within [2^-10, 2688] and is exact in f16; an E4M3 value is exact in
// f16 (the window's float32 row scale multiplies its scores and its P instead).
#include <cfloat>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace csa2 {

constexpr int kTcChunk = 128;            // key rows per step (N of S, K of P V)
constexpr int kTcMaxH = 64;              // heads per row (M of both products)
constexpr int kWsThreads = 13 * 32;      // softmax warps 0-7, producer warps 8-11, MMA warp 12
constexpr int kWsMmaWarp = 12;
constexpr int kWsProdWarp0 = 8;
constexpr int kWsRaw = 3;                // raw gather stages per producer thread
constexpr int kWsK = 3;                  // f16 key stages
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
constexpr int kOffP = kOffK + kWsK * kKBytes;
constexpr int kOffRaw = kOffP + 2 * kPBytes;
constexpr int kOffKf = kOffRaw + kWsRaw * kRawStage;      // [K stage][kmul | kval][128] float
constexpr int kOffUni = kOffKf + kWsK * 2 * kTcChunk * 4; // [K stage][4 producer warps] int
constexpr int kWsSmem = kOffUni + kWsK * 4 * 4;
static_assert(kWsSmem <= 226 * 1024, "one CTA per SM");
constexpr int kWsCols = 512;             // TMEM columns: S buffers at 0 and 128, O buffers at 256 and 384

// mbarriers; the k-th completion of a barrier of stage x (of n stages) belongs to step (or
// row) x + n k, so its phase parity is k & 1
enum {
  kBarKFull = 0,     // [3] keys of a step (at a row's first step also its queries) in: 4 producer-warp arrivals
  kBarKEmpty = 3,    // [3] P V of the step in a K stage complete: MMA commit
  kBarSFull = 6,     // [2] S of a step in its TMEM buffer: MMA commit
  kBarPFull = 8,     // [2] P of a step written and O rescaled: 8 softmax-warp arrivals
  kBarPvDone = 10,   // [2] P V of a step complete: MMA commit
  kBarQEmpty = 12,   // [2] every S of a row complete (its Q stage is free): MMA commit
  kBarOEmpty = 14,   // [2] a row's O buffer read out: 8 softmax-warp arrivals
  kBarFin = 16,      // every MMA issued has completed
  kNumBars = 17
};
__host__ __device__ constexpr int bar_count(int i) {
  return i < kBarKEmpty ? 4 : ((i >= kBarPFull && i < kBarPvDone) || (i >= kBarOEmpty && i < kBarFin)) ? 8 : 1;
}

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

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}
// packed two-wide float32 arithmetic (one instruction for a key pair; each half rounds as
// the scalar operation would)
__device__ __forceinline__ uint64_t f2_bits(float2 a) { return ((uint64_t)__float_as_uint(a.y) << 32) | __float_as_uint(a.x); }
__device__ __forceinline__ float2 bits_f2(uint64_t r) {
  return make_float2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(r);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(r);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(r);
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

// 64 TMEM columns of 16 lanes, 16x256b shape: thread t gets lane t / 4 (r[4 j], r[4 j + 1])
// and lane t / 4 + 8 (r[4 j + 2], r[4 j + 3]), columns 8 j + 2 (t % 4) and + 1.  The wait
// is a separate statement that every use of the registers depends on.
__device__ __forceinline__ void tmem_ld64c(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_st64c(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__global__ void __launch_bounds__(kWsThreads, 1) attn_chunked_tc_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(16) uint8_t s_dyn[];
  __shared__ __align__(8) uint64_t s_bar[kNumBars];
  __shared__ uint32_t s_tmem;
  __shared__ float2 s_xm[2][8][32];                          // softmax pairs: step maxima, by step parity
  __shared__ float2 s_xl[8][32];                             //   and row sums at a row's end
  __shared__ __align__(8) uint64_t s_xbar[4][4];             // their exchanges: [pair][step parity, row parity]
  pdl_enter();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t G = gridDim.x;
  const int64_t nrows = a.T > (int64_t)blockIdx.x ? (a.T - 1 - (int64_t)blockIdx.x) / G + 1 : 0;
  const int NC = a.n_chunks;
  const int64_t U = nrows * NC;                              // (row, chunk) steps of this CTA
  auto bar = [&](int i) { return smem_addr(&s_bar[i]); };

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar(i)), "r"(bar_count(i)));
    for (int i = 0; i < 16; ++i)                           // two warp arrivals each
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;\n" ::"r"(smem_addr(&s_xbar[i >> 2][i & 3])));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == kWsMmaWarp) {
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

  if (warp == kWsMmaWarp) {
    // ================================================================ MMA issue (one thread)
    if (lane == 0 && U > 0) {
      const uint32_t id_s = umma_idesc(kTcMaxH, kTcChunk, 0, 0);   // S = Q K^T: A, B K-major
      const uint32_t id_o = umma_idesc(kTcMaxH, kD, 0, 1);         // O += P V: A K-major, B MN-major
      const uint32_t q_a = smem_addr(s_dyn + kOffQ), k_a = smem_addr(s_dyn + kOffK), p_a = smem_addr(s_dyn + kOffP);
      // P V of step v (row iv, chunk cv, K stage kv); the descriptors advance 16 keys per MMA
      auto issue_pv = [&](int64_t v, int64_t iv, int cv, int kv) -> bool {
        const int x = (int)(v & 1);
        if (cv == 0 && iv >= 2 && !mbar_wait(bar(kBarOEmpty + (int)(iv & 1)), (uint32_t)(((iv - 2) >> 1) & 1)))
          return false;
        if (!mbar_wait(bar(kBarPFull + x), (uint32_t)((v >> 1) & 1))) return false;
        tc_fence_after();
        const uint32_t d = tmem + 256 + 128 * (uint32_t)(iv & 1);
        const uint64_t dp = umma_desc(p_a + x * kPBytes, 128, 2048), dv = umma_desc(k_a + kv * kKBytes, 2048, 128);
#pragma unroll
        for (int s = 0; s < kTcChunk / 16; ++s)
          umma_f16(d, dp + (uint64_t)(16 * s), dv + (uint64_t)(256 * s), id_o, (cv > 0 || s > 0) ? 1u : 0u);
        umma_commit(bar(kBarPvDone + x));
        umma_commit(bar(kBarKEmpty + kv));
        return true;
      };
      int64_t i = 0, pi = 0;
      int c = 0, pc = 0, ks = 0, pks = 0;                    // (row, chunk, K stage) of steps u and u - 1
      uint32_t kph = 0;                                      // phase parity of step u on its K stage
      for (int64_t u = 0; u < U; ++u) {
        const int x = (int)(u & 1);
        if (!mbar_wait(bar(kBarKFull + ks), kph)) { dead = true; break; }
        tc_fence_after();
        const uint64_t dq = umma_desc(q_a + (uint32_t)(i & 1) * kQBytes, 128, 2048);
        const uint64_t dk = umma_desc(k_a + ks * kKBytes, 128, 2048);
#pragma unroll
        for (int s = 0; s < kD / 16; ++s)
          umma_f16(tmem + 128 * (uint32_t)x, dq + (uint64_t)(16 * s), dk + (uint64_t)(16 * s), id_s, s > 0 ? 1u : 0u);
        umma_commit(bar(kBarSFull + x));
        if (c == NC - 1) umma_commit(bar(kBarQEmpty + (int)(i & 1)));
        if (u >= 1 && !issue_pv(u - 1, pi, pc, pks)) { dead = true; break; }
        pi = i;
        pc = c;
        pks = ks;
        if (++c == NC) { c = 0; ++i; }
        if (++ks == kWsK) { ks = 0; kph ^= 1u; }
      }
      if (!dead) dead = !issue_pv(U - 1, pi, pc, pks);
      // every MMA issued has completed before TMEM is released
      umma_commit(bar(kBarFin));
      if (!mbar_wait(bar(kBarFin), 0)) dead = true;
    }
  } else if (warp >= kWsProdWarp0) {
    // ================================================================ producers
    const int pt = tid - 32 * kWsProdWarp0, pw = pt >> 5;                  // key row pt of every step
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
    auto issue = [&](int64_t v, int slot) {
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
    for (int s = 0; s < kWsRaw; ++s) issue(s, s);

    int64_t i = 0;
    int c = 0, ks = 0, slot = 0;
    uint32_t kph = 0;                                        // phase parity of step u on its K stage
    for (int64_t u = 0; u < U; ++u) {
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
      // K stage ks is free once the P V of step u - 3 is complete
      if (u >= kWsK && !mbar_wait_warp(bar(kBarKEmpty + ks), kph ^ 1u)) { dead = true; break; }
      const bool valid = (vbits >> slot) & 1u, fp8 = (fbits >> slot) & 1u;
      uint8_t *kt = s_dyn + kOffK + ks * kKBytes + krow;
      const uint8_t *raw = raw_g + slot * kRawStage;
      float kmul = 0.f, kval = -1.f;
      if (!valid) {
#pragma unroll
        for (int dg = 0; dg < 16; ++dg) *reinterpret_cast<uint4 *>(kt + dg * 128) = make_uint4(0, 0, 0, 0);
      } else if (!fp8) {
        const uint2 sc = *reinterpret_cast<const uint2 *>(raw + 128);
        const uint4 c0 = *reinterpret_cast<const uint4 *>(raw), c1 = *reinterpret_cast<const uint4 *>(raw + 16);
        const uint4 c2 = *reinterpret_cast<const uint4 *>(raw + 32), c3 = *reinterpret_cast<const uint4 *>(raw + 48);
        const uint32_t cw[16] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w,
                                 c2.x, c2.y, c2.z, c2.w, c3.x, c3.y, c3.z, c3.w};
        uint32_t sp[4];                                      // the eight group scales as f16 pairs
        e4m3x4_to_f16(sc.x, sp[0], sp[1]);
        e4m3x4_to_f16(sc.y, sp[2], sp[3]);
#pragma unroll
        for (int g = 0; g < 8; ++g) {                        // channels 16 g .. 16 g + 15: two core-matrix rows
          const uint32_t sh = (g & 1) ? (sp[g >> 1] >> 16) : (sp[g >> 1] & 0xFFFFu);
          const uint32_t s2 = sh | (sh << 16);
          uint32_t lo[4], hi[4], v[8];
          e2m1x8_to_f16(cw[2 * g], lo);
          e2m1x8_to_f16(cw[2 * g + 1], hi);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[e] = hmul2_bits(lo[e], s2);
            v[4 + e] = hmul2_bits(hi[e], s2);
          }
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
          uint32_t v[8];
          e4m3x4_to_f16(w.x, v[0], v[1]);
          e4m3x4_to_f16(w.y, v[2], v[3]);
          e4m3x4_to_f16(w.z, v[4], v[5]);
          e4m3x4_to_f16(w.w, v[6], v[7]);
          *reinterpret_cast<uint4 *>(kt + (2 * g) * 128) = make_uint4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<uint4 *>(kt + (2 * g + 1) * 128) = make_uint4(v[4], v[5], v[6], v[7]);
        }
        kmul = ltau * wsc;
        kval = wsc;
      }
      kf[ks * 2 * kTcChunk + pt] = kmul;
      kf[ks * 2 * kTcChunk + kTcChunk + pt] = kval;
      const bool uni = __all_sync(0xffffffffu, valid && !fp8);
      if (lane == 0) kuni[ks * 4 + pw] = uni ? 1 : 0;
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarKFull + ks));
      issue(u + kWsRaw, slot);                               // the raw stage is free again
      if (++c == NC) { c = 0; ++i; }
      if (++ks == kWsK) { ks = 0; kph ^= 1u; }
      if (++slot == kWsRaw) slot = 0;
    }
    cp_async_wait<0>();
  } else {
    // ================================================================ softmax (warps 0-7)
    // warp w reads the TMEM lanes of quarter w & 3 (heads 16 (w & 3) .. + 15) and takes key
    // half kh = w >> 2 of every step (key groups 8 kh .. 8 kh + 7) and output dims 64 kh ..
    // 64 kh + 63; warps w and w ^ 4 share their heads' step maxima and row sums
    const int wq = warp & 3, kh = warp >> 2, q4 = lane & 3;
    const int h0 = 16 * wq + (lane >> 2), h1 = h0 + 8;      // this thread's two heads
    const bool own0 = h0 < a.H, own1 = h1 < a.H;
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    const float *kf = reinterpret_cast<const float *>(s_dyn + kOffKf);
    const int *kuni = reinterpret_cast<const int *>(s_dyn + kOffUni);
    const float ltau = a.tau * kTcLog2e;
    // P rows of the two heads: core matrix (head group, key group 8 kh + g), row head % 8, word q4
    const int p0off = (h0 >> 3) * 2048 + 8 * kh * 128 + (h0 & 7) * 16 + 4 * q4, p1off = p0off + 2048;
    // exchange with the partner warp: this warp's values are stored; arrive, then a bounded
    // wait for the partner's arrival on the same phase (k-th completion of slot x: step or
    // row x + 2 k)
    auto pair_sync = [&](int slot, int64_t n) -> bool {
      const uint32_t b = smem_addr(&s_xbar[wq][slot]);
      __syncwarp();
      if (lane == 0) mbar_arrive(b);
      return mbar_wait_warp(b, (uint32_t)((n >> 1) & 1));
    };
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int64_t i = 0;
    int c = 0, ks = 0;
    uint32_t kph = 0;
    for (int64_t u = 0; u < U; ++u) {
      const int x = (int)(u & 1);
      const uint32_t par = (uint32_t)((u >> 1) & 1);
      if (!mbar_wait_warp(bar(kBarKFull + ks), kph) || !mbar_wait_warp(bar(kBarSFull + x), par)) { dead = true; break; }
      tc_fence_after();
      // s[2 g], s[2 g + 1]: head h0, keys 8 (8 kh + g) + 2 q4 and + 1; s[16 + ...]: head h1
      float s[32];
      {
        uint32_t r[32];
        tmem_ld64c(tmem + lane_base + 128 * (uint32_t)x + 64 * kh, r);
        tmem_ld_wait32(r);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          s[2 * g] = __uint_as_float(r[4 * g]);
          s[2 * g + 1] = __uint_as_float(r[4 * g + 1]);
          s[16 + 2 * g] = __uint_as_float(r[4 * g + 2]);
          s[16 + 2 * g + 1] = __uint_as_float(r[4 * g + 3]);
        }
      }
      const int4 un = *reinterpret_cast<const int4 *>(kuni + 4 * ks);
      const bool uni = un.x && un.y && un.z && un.w;         // every key a valid top-k row
      const float *km = kf + ks * 2 * kTcChunk + 64 * kh, *kv = km + kTcChunk;
      // per head: the maximum of this key half over four partial maxima and the quad, then
      // over the partner warp's half
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
      if (uni) {
        const float2 lt2 = make_float2(ltau, ltau);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float2 z = mul2(make_float2(s[j], s[j + 1]), lt2);
          s[j] = z.x;
          s[j + 1] = z.y;
          mx[(j >> 4) * 4 + (j & 3)] = fmaxf(mx[(j >> 4) * 4 + (j & 3)], z.x);
          mx[(j >> 4) * 4 + ((j + 1) & 3)] = fmaxf(mx[(j >> 4) * 4 + ((j + 1) & 3)], z.y);
        }
      } else {
#pragma unroll
        for (int g = 0; g < 8; ++g) {                        // key pair 8 (8 kh + g) + 2 q4, + 1
          const float2 f = *reinterpret_cast<const float2 *>(km + 8 * g + 2 * q4);
          const float2 v = *reinterpret_cast<const float2 *>(kv + 8 * g + 2 * q4);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int j = 16 * hh + 2 * g;
            s[j] = v.x >= 0.f ? s[j] * f.x : -INFINITY;
            s[j + 1] = v.y >= 0.f ? s[j + 1] * f.y : -INFINITY;
            mx[4 * hh + (j & 3)] = fmaxf(mx[4 * hh + (j & 3)], s[j]);
            mx[4 * hh + ((j + 1) & 3)] = fmaxf(mx[4 * hh + ((j + 1) & 3)], s[j + 1]);
          }
        }
      }
      float cm0 = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      float cm1 = fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, 1));
      cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, 1));
      cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, 2));
      cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, 2));
      s_xm[x][warp][lane] = make_float2(cm0, cm1);
      if (!pair_sync(x, u)) { dead = true; break; }
      {
        const float2 o = s_xm[x][warp ^ 4][lane];
        cm0 = fmaxf(cm0, o.x);
        cm1 = fmaxf(cm1, o.y);
      }
      // the reference maxima: the step's at a row's start, later raised past 2^8 only (both
      // warps of a pair take the same decisions)
      bool r0 = false, r1 = false;
      float al0 = 1.f, al1 = 1.f;
      if (c == 0) {
        m0 = cm0;
        m1 = cm1;
        l0 = 0.f;
        l1 = 0.f;
      } else {
        if (cm0 > m0 + kRescaleLog2 || (m0 == -INFINITY && cm0 > -INFINITY)) {
          r0 = true;
          al0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - cm0);
          m0 = cm0;
        }
        if (cm1 > m1 + kRescaleLog2 || (m1 == -INFINITY && cm1 > -INFINITY)) {
          r1 = true;
          al1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - cm1);
          m1 = cm1;
        }
      }
      // P stage x is free once the P V of step u - 2 is complete
      if (u >= 2 && !mbar_wait_warp(bar(kBarPvDone + x), (uint32_t)(((u - 2) >> 1) & 1))) { dead = true; break; }
      // P of the two heads (f16, times the window rows' scales) into the A operand; the row
      // sums add the unrounded values
      uint8_t *ps = s_dyn + kOffP + x * kPBytes;
      float2 la[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};                // partial sums [head][parity of g], per pair
      const float2 m0p = make_float2(m0, m0), m1p = make_float2(m1, m1);
      if (uni) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int j = 16 * hh + 2 * g;
            const float2 d = sub2(make_float2(s[j], s[j + 1]), hh ? m1p : m0p);
            const float2 pp = make_float2(ex2_approx(d.x), ex2_approx(d.y));
            la[2 * hh + (g & 1)] = add2(la[2 * hh + (g & 1)], pp);
            *reinterpret_cast<uint32_t *>(ps + (hh ? p1off : p0off) + g * 128) = pack_f16x2(pp.x, pp.y);
          }
        }
      } else {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float2 v = *reinterpret_cast<const float2 *>(kv + 8 * g + 2 * q4);
          const float2 vv = make_float2(fmaxf(v.x, 0.f), fmaxf(v.y, 0.f));
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int j = 16 * hh + 2 * g;
            const float2 d = sub2(make_float2(s[j], s[j + 1]), hh ? m1p : m0p);
            const float2 pp = make_float2(s[j] == -INFINITY ? 0.f : ex2_approx(d.x),
                                          s[j + 1] == -INFINITY ? 0.f : ex2_approx(d.y));
            la[2 * hh + (g & 1)] = add2(la[2 * hh + (g & 1)], pp);
            const float2 pv = mul2(pp, vv);
            *reinterpret_cast<uint32_t *>(ps + (hh ? p1off : p0off) + g * 128) = pack_f16x2(pv.x, pv.y);
          }
        }
      }
      {
        const float2 s0 = add2(la[0], la[1]), s1 = add2(la[2], la[3]);
        l0 = l0 * al0 + (s0.x + s0.y);
        l1 = l1 * al1 + (s1.x + s1.y);
      }
      // a head's reference maximum rose: rescale this warp's half of its O row once the P V
      // of step u - 1 is in (the TMEM access is warp-wide, so the warp rescales when any of
      // its heads needs it)
      if (__any_sync(0xffffffffu, r0 || r1)) {
        if (!mbar_wait_warp(bar(kBarPvDone + (x ^ 1)), (uint32_t)(((u - 1) >> 1) & 1))) { dead = true; break; }
        tc_fence_after();
        const uint32_t t_o = tmem + lane_base + 256 + 128 * (uint32_t)(i & 1) + 64 * kh;
        uint32_t r[32];
        tmem_ld64c(t_o, r);
        tmem_ld_wait32(r);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) * al0);
          r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) * al0);
          r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) * al1);
          r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) * al1);
        }
        tmem_st64c(t_o, r);
        tmem_st_wait();
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + x));
      if (c == NC - 1) {
        // ---- the row's end: O / l and the log-sum-exp, then its O buffer is free
        float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
        float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
        s_xl[warp][lane] = make_float2(lt0, lt1);
        if (!pair_sync(2 + (int)(i & 1), i)) { dead = true; break; }
        {
          const float2 o = s_xl[warp ^ 4][lane];
          lt0 += o.x;
          lt1 += o.y;
        }
        if (!mbar_wait_warp(bar(kBarPvDone + x), par)) { dead = true; break; }
        tc_fence_after();
        const int64_t t = (int64_t)blockIdx.x + i * G;
        const float inv0 = lt0 > 0.f ? 1.f / lt0 : 0.f, inv1 = lt1 > 0.f ? 1.f / lt1 : 0.f;
        const uint32_t t_o = tmem + lane_base + 256 + 128 * (uint32_t)(i & 1) + 64 * kh;
        float *o0 = a.out + (t * a.H + (own0 ? h0 : 0)) * kD + 64 * kh + 2 * q4;
        float *o1 = a.out + (t * a.H + (own1 ? h1 : 0)) * kD + 64 * kh + 2 * q4;
        uint32_t r[32];
        tmem_ld64c(t_o, r);
        tmem_ld_wait32(r);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (own0)
            *reinterpret_cast<float2 *>(o0 + 8 * j) =
                make_float2(__uint_as_float(r[4 * j]) * inv0, __uint_as_float(r[4 * j + 1]) * inv0);
          if (own1)
            *reinterpret_cast<float2 *>(o1 + 8 * j) =
                make_float2(__uint_as_float(r[4 * j + 2]) * inv1, __uint_as_float(r[4 * j + 3]) * inv1);
        }
        if (kh == 0 && q4 == 0 && a.lse) {
          if (own0) a.lse[t * a.H + h0] = lt0 > 0.f ? m0 / kTcLog2e + logf(lt0) : -INFINITY;
          if (own1) a.lse[t * a.H + h1] = lt1 > 0.f ? m1 / kTcLog2e + logf(lt1) : -INFINITY;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarOEmpty + (int)(i & 1)));
      }
      if (++c == NC) { c = 0; ++i; }
      if (++ks == kWsK) { ks = 0; kph ^= 1u; }
    }
  }
  if (dead) set_err(a.d_err, CSA2_DEVERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWsMmaWarp) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kWsCols));
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
