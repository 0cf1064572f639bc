// kv_append_fp4: RoPE + FP4 (E2M1 / E4M3 per 16 channels) main KV, FP8 indexer
// key, FP8 SWA ring.  One warp per (token, part): part 0 writes the main KV row and the
// indexer key, part 1 + l the token's row of SWA layer l.  Every load a warp needs is
// issued before it waits on any of them.
// Method: origotech.dev deep dive, subsection "FP4와 SWA Bounded Replay" (FP4
// main KV quantised after RoPE, SWA KV in FP8).
#include "common.cuh"
#include "launch.h"

namespace csa2 {

// r0 = x0*c - x1*s, r1 = x0*s + x1*c with every operation rounded on its own
__device__ __forceinline__ void rotate(float &x0, float &x1, float c, float s) {
  float r0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
  float r1 = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
  x0 = r0;
  x1 = r1;
}

// FP4 code of one value given its group's decoded scale s (sign bit copied from v)
__device__ __forceinline__ uint32_t fp4_code(float v, float s) {
  uint32_t mag = (s > 0.f) ? f32_to_e2m1_mag(__fdiv_rn(fabsf(v), s)) : 0u;
  return mag | ((__float_as_uint(v) >> 28) & 8u);
}

// FP8 code of one value given the row's float32 scale s
__device__ __forceinline__ uint32_t fp8_code(float v, float s) {
  return (s > 0.f) ? f32_to_e4m3(__fdiv_rn(v, s)) : 0u;
}

// 4 consecutive channels per lane; a 16-channel group spans 4 lanes.
// Returns the 2 packed code bytes (low byte = first two channels) and the
// group's scale code in *scode.
__device__ __forceinline__ uint32_t quant_fp4_lane(float x[4], uint32_t *scode) {
  float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  uint32_t sc = f32_to_e4m3(__fdiv_rn(a, 6.0f));
  float s = e4m3_to_f32(sc);
  *scode = sc;
  uint32_t c0 = fp4_code(x[0], s), c1 = fp4_code(x[1], s), c2 = fp4_code(x[2], s), c3 = fp4_code(x[3], s);
  return (c0 | (c1 << 4)) | ((c2 | (c3 << 4)) << 8);
}

struct AppendArgs {
  csa2_cache c;
  csa2_swa swa[CSA2_MAX_SWA_LAYERS];
  int32_t n_swa;
  const uint16_t *kv_new, *ik_new, *swa_new;
  const float *cos, *sin;
  int64_t rope_len;
  const int32_t *seq_id;
  const int64_t *pos;
  int64_t n;
  int32_t main_part;       // 1: part 0 writes the main KV (+ indexer key); 0: window rings only
  int32_t *d_err;
};

__device__ __forceinline__ void load4_bf16(const uint16_t *p, float x[4]) {
  uint2 raw = __ldg(reinterpret_cast<const uint2 *>(p));
  x[0] = bf16_to_f32(raw.x & 0xFFFFu);
  x[1] = bf16_to_f32(raw.x >> 16);
  x[2] = bf16_to_f32(raw.y & 0xFFFFu);
  x[3] = bf16_to_f32(raw.y >> 16);
}

__global__ void __launch_bounds__(256) kv_append_kernel(const __grid_constant__ AppendArgs a) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int parts = (a.swa_new ? a.n_swa : 0) + a.main_part;
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t tok = wid / parts;
  const int part = (int)(wid - tok * parts) + 1 - a.main_part;   // 0 = main KV, 1 + l = window layer l
  if (tok >= a.n) return;
  // independent loads first: the token's identity and this part's input row
  const int b = __ldg(a.seq_id + tok);
  const int64_t p = __ldg(a.pos + tok);
  const uint16_t *src = part == 0 ? a.kv_new + tok * kD : a.swa_new + ((int64_t)(part - 1) * a.n + tok) * kD;
  const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(src + 4 * lane));
  uint32_t ik_raw = 0;
  if (part == 0 && a.ik_new) ik_raw = __ldg(reinterpret_cast<const uint32_t *>(a.ik_new + tok * kDIdx + 2 * lane));
  if (b < 0 || b >= a.c.B) {
    if (lane == 0) set_err(a.d_err, CSA2_DEVERR_SEQ);
    return;
  }
  if (p < 0 || p >= a.rope_len) {
    if (lane == 0) set_err(a.d_err, CSA2_DEVERR_POS);
    return;
  }
  // rotation operands of this lane's channel pairs (lanes 16..31 hold channels 64..127)
  float c0 = 1.f, s0 = 0.f, c1 = 1.f, s1 = 0.f;
  if (lane >= 16) {
    const int i0 = 2 * lane - 32;
    const float *cr = a.cos + p * (kDRope / 2), *sr = a.sin + p * (kDRope / 2);
    c0 = __ldg(cr + i0); s0 = __ldg(sr + i0);
    c1 = __ldg(cr + i0 + 1); s1 = __ldg(sr + i0 + 1);
  }
  float x[4] = {bf16_to_f32(raw.x & 0xFFFFu), bf16_to_f32(raw.x >> 16), bf16_to_f32(raw.y & 0xFFFFu),
                bf16_to_f32(raw.y >> 16)};
  if (lane >= 16) { rotate(x[0], x[1], c0, s0); rotate(x[2], x[3], c1, s1); }

  // a token whose cache row is out of range is skipped by every part
  const int64_t row = a.main_part ? a.c.seq_base[b] + p : 0;
  if (a.main_part && (row < 0 || row >= a.c.T_cap)) {
    if (lane == 0) set_err(a.d_err, CSA2_DEVERR_POS);
    return;
  }
  if (part == 0) {
    // main KV -> FP4
    uint32_t scode;
    uint32_t packed = quant_fp4_lane(x, &scode);
    *reinterpret_cast<uint16_t *>(a.c.kv_codes + row * (kD / 2) + 2 * lane) = (uint16_t)packed;
    if ((lane & 3) == 0) a.c.kv_scales[row * (kD / 16) + (lane >> 2)] = (uint8_t)scode;
    // indexer key -> FP8 with a per-token scale (no rotation)
    if (a.ik_new) {
      float x0 = bf16_to_f32(ik_raw & 0xFFFFu), x1 = bf16_to_f32(ik_raw >> 16);
      float am = warp_max(fmaxf(fabsf(x0), fabsf(x1)));
      float s = __fdiv_rn(am, 448.0f);
      uint32_t code = fp8_code(x0, s) | (fp8_code(x1, s) << 8);
      *reinterpret_cast<uint16_t *>(a.c.ik_codes + row * kDIdx + 2 * lane) = (uint16_t)code;
      if (lane == 0) a.c.ik_scale[row] = s;
    }
  } else {
    // SWA layer part - 1: rotated like the main KV, FP8 with a per-token scale, ring slot p % ring
    float am = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
    float s = __fdiv_rn(am, 448.0f);
    uint32_t code = fp8_code(x[0], s) | (fp8_code(x[1], s) << 8) | (fp8_code(x[2], s) << 16) |
                    (fp8_code(x[3], s) << 24);
    const csa2_swa &w = a.swa[part - 1];
    const int64_t slot = (int64_t)b * w.ring + (p % w.ring);
    *reinterpret_cast<uint32_t *>(w.codes + slot * kD + 4 * lane) = code;
    if (lane == 0) w.scale[slot] = s;
  }
}

cudaError_t launch_append(const csa2_cache &c, const csa2_swa *swa, int n_swa, const uint16_t *kv_new,
                          const uint16_t *ik_new, const uint16_t *swa_new, const float *cos,
                          const float *sin, int64_t rope_len, const int32_t *seq_id, const int64_t *pos,
                          int64_t n, int32_t *d_err, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  AppendArgs a;
  a.c = c;
  for (int l = 0; l < n_swa; ++l) a.swa[l] = swa[l];
  for (int l = n_swa; l < CSA2_MAX_SWA_LAYERS; ++l) a.swa[l] = csa2_swa{nullptr, nullptr, 1};
  a.n_swa = n_swa;
  a.kv_new = kv_new; a.ik_new = ik_new; a.swa_new = swa_new;
  a.cos = cos; a.sin = sin; a.rope_len = rope_len;
  a.seq_id = seq_id; a.pos = pos; a.n = n; a.d_err = d_err;
  a.main_part = kv_new ? 1 : 0;
  const int warps = 8;
  const int64_t parts = (swa_new ? n_swa : 0) + a.main_part;
  if (parts == 0) return cudaSuccess;
  const int64_t grid = (n * parts + warps - 1) / warps;
  return launch_k(kv_append_kernel, dim3((unsigned)grid), dim3(warps * 32), 0, st, 0, a);
}

// ---- test-only kernels: the same quantisers on raw float32 data ----

__global__ void test_fp4_kernel(const float *x, int64_t n_groups, uint8_t *codes, uint8_t *scales) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  // one warp handles 8 groups: lanes 4k..4k+3 hold group w*8+k
  const int64_t g = w * 8 + (lane >> 2);
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  const bool ok = g < n_groups;
  if (ok) {
    float4 f = *reinterpret_cast<const float4 *>(x + g * 16 + 4 * (lane & 3));
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  }
  uint32_t scode;
  uint32_t packed = quant_fp4_lane(v, &scode);
  if (ok) {
    *reinterpret_cast<uint16_t *>(codes + g * 8 + 2 * (lane & 3)) = (uint16_t)packed;
    if ((lane & 3) == 0) scales[g] = (uint8_t)scode;
  }
}

__global__ void test_fp8_kernel(const float *x, int64_t n, int C, uint8_t *codes, float *scale) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= n) return;
  const int per = C / 32;  // 2 or 4 values per lane
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  float am = 0.f;
  for (int i = 0; i < per; ++i) { v[i] = x[r * C + per * lane + i]; am = fmaxf(am, fabsf(v[i])); }
  am = warp_max(am);
  float s = __fdiv_rn(am, 448.0f);
  for (int i = 0; i < per; ++i) codes[r * C + per * lane + i] = (uint8_t)fp8_code(v[i], s);
  if (lane == 0) scale[r] = s;
}

cudaError_t launch_test_fp4(const float *x, int64_t n_groups, uint8_t *codes, uint8_t *scales,
                            cudaStream_t st) {
  if (n_groups == 0) return cudaSuccess;
  const int64_t warps = (n_groups + 7) / 8;
  test_fp4_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(x, n_groups, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_test_fp8(const float *x, int64_t n, int C, uint8_t *codes, float *scale, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  test_fp8_kernel<<<(unsigned)((n + 7) / 8), 256, 0, st>>>(x, n, C, codes, scale);
  return cudaGetLastError();
}

}  // namespace csa2
