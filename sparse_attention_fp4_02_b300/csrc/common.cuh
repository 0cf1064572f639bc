// Shared device helpers of the CSA2 library (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_fp4.h>

#include "csa2.h"

namespace csa2 {

constexpr int kD = CSA2_D;
constexpr int kDRope = CSA2_D_ROPE;
constexpr int kDIdx = CSA2_D_IDX;
constexpr int kHIdx = CSA2_H_IDX;
constexpr int kHistBins = 4096;      // top 12 bits of a non-negative float32
constexpr int kHistShift = 19;

__device__ __forceinline__ void set_err(int32_t *d_err, int bits) { atomicOr(d_err, bits); }

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// float -> E4M3, round to nearest even, saturating to +-448
__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
  return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(__half(h));
}

// two E4M3 codes (low byte -> low half) to a packed f16x2; exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xFFFFu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// eight E2M1 codes (a 32-bit word, low nibble first) to four packed f16 pairs; exact
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n .reg .b8 c0, c1, c2, c3;\n mov.b32 {c0, c1, c2, c3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, c0;\n cvt.rn.f16x2.e2m1x2 %1, c1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, c2;\n cvt.rn.f16x2.e2m1x2 %3, c3;\n}\n"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

// four E4M3 codes (low byte first) to two packed f16 pairs; exact
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t &o0, uint32_t &o1) {
  asm("{\n .reg .b16 h0, h1;\n mov.b32 {h0, h1}, %2;\n cvt.rn.f16x2.e4m3x2 %0, h0;\n cvt.rn.f16x2.e4m3x2 %1, h1;\n}\n"
      : "=r"(o0), "=r"(o1)
      : "r"(w));
}

// 2^x from the special-function unit (ex2.approx, relative error near 2^-22); flushes
// subnormal results to zero
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// non-negative float -> E2M1 magnitude code 0..7, nearest even, saturating at 6
__device__ __forceinline__ uint32_t f32_to_e2m1_mag(float x) {
  return (uint32_t)__nv_cvt_float_to_fp4(x, __NV_E2M1, cudaRoundNearest) & 7u;
}

// Power-of-two shift c that brings a query head whose largest |value| is mx into f16 with
// its maximum in [2^14, 2^15): every value above 2^-29 of the maximum stays exact.
__device__ __forceinline__ int head_shift(float mx) {
  if (!(mx > 0.f)) return 0;
  int e = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;
  int c = 14 - e;
  return c < -60 ? -60 : (c > 60 ? 60 : c);
}

__device__ __forceinline__ float pow2f(int c) { return __uint_as_float((uint32_t)(c + 127) << 23); }

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// D += A * B, m16n8k16, f16 inputs, f32 accumulate
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                        const void *smem_row) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(smem_row);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                          const void *smem_row) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(smem_row);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}

// streaming 16-byte load that bypasses L1
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_nc16(const void *p) {
  return __ldg(reinterpret_cast<const uint4 *>(p));
}

// cp.async copies into shared memory; pred false zero-fills without reading the source
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(pred ? 16 : 0));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, bool pred) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(pred ? 4 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
// TMA bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from global to
// shared memory, completing the transaction count of the mbarrier at `mbar`
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(mbar)
               : "memory");
}
// arrive on the mbarrier and add `bytes` to the transaction count its phase waits for
__device__ __forceinline__ void mbar_expect_tx_u32(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(mbar), "r"(bytes) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// Programmatic dependent launch: a kernel launched with launch_k may be scheduled while
// the previous kernel in the stream finishes.  Each kernel first waits for that kernel
// (and so, transitively, for every earlier one) to complete and publish its memory, then
// lets the next kernel be scheduled.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_trigger();
}

// Launch with programmatic stream serialisation (and, if cluster_x > 0, that cluster size).
template <class Kernel, class... Args>
cudaError_t launch_k(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, unsigned cluster_x,
                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace csa2
