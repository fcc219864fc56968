// Device helpers shared by the decode-step kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/mbt.h"

namespace mbt {

typedef __nv_bfloat16 bf16;

constexpr int kBlockTokens = 16;     // tokens per paged KV block

enum WType { W_BF16 = 0, W_E4M3 = 1 };

// ---------------------------------------------------------------------------
// global memory

// 16-byte streaming load of data read exactly once (weights): bypass L1.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Programmatic dependent launch: let the next kernel of the stream start its
// independent prologue now, and wait for the previous kernel's results. Both
// are no-ops for a kernel launched without the PDL attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Pull read-only bytes into L2 ahead of use (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void set_err(uint32_t* err, uint32_t bit) {
  if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------------------
// number formats

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two e4m3 codes (low byte first) -> two floats, exactly (hardware conversion
// to f16, which holds every e4m3 value, then to f32).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xffffu), __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// Two e4m3 codes (low byte first) -> FP16x2 bits, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_h2bits(uint32_t two_codes) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xffffu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// x = hi + lo in the 16-bit format the next tensor-core projection reads.
__device__ __forceinline__ void store_hl16(uint16_t* hi_at, uint16_t* lo_at, float x, int f16) {
  if (f16) {
    const __half h = __float2half_rn(x);
    *hi_at = __half_as_ushort(h);
    *lo_at = __half_as_ushort(__float2half_rn(x - __half2float(h)));
  } else {
    const bf16 h = __float2bfloat16_rn(x);
    *hi_at = __bfloat16_as_ushort(h);
    *lo_at = __bfloat16_as_ushort(__float2bfloat16_rn(x - __bfloat162float(h)));
  }
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3)));
}

// Activation rows for e4m3 x e4m3 tensor-core products: four e4m3 terms per
// value, x = s * (c0 + c1 / 16 + c2 / 256 + c3 / 4096) + e, with s a power of
// two per row such that max |x| / s < 448. Each step rounds the scaled residual
// to e4m3 and carries the rest, times 16, to the next code; the residual is
// exact in fp32 (a rounding to the nearest e4m3 value is within a factor
// 1 +- 1/16 of the value, or on a grid no finer than the value's own), so
// |e| <= |x| / 2^16 plus, for values far below the row's largest, s / 2^22.
constexpr int kTerms = 4;

// Scale of a row whose largest magnitude is m: s = 2^e with m / s in [224, 448);
// 1 for an all-zero row; NaN when m is not finite (the products then carry it).
__device__ __forceinline__ void term_scale(float m, float& s, float& inv) {
  if (!(m <= 3.0e38f)) { s = inv = __int_as_float(0x7fc00000); return; }
  if (m == 0.f) { s = inv = 1.f; return; }
  int e;
  frexpf(m * (1.f / 448.f), &e);
  s = ldexpf(1.f, e);
  inv = ldexpf(1.f, -e);
}

// The four codes of x (term j in byte j) given 1 / s.
__device__ __forceinline__ uint32_t split_terms(float x, float inv_s) {
  float r = x * inv_s;
  uint32_t out = 0;
#pragma unroll
  for (int j = 0; j < kTerms; ++j) {
    const uint32_t c = f32_to_e4m3(r);
    out |= c << (8 * j);
    r = (r - e4m3_to_f32(c)) * 16.f;
  }
  return out;
}

// ---------------------------------------------------------------------------
// reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024). `scratch` holds
// >= 32 floats. Every thread returns the total.
// ---------------------------------------------------------------------------
// thread-block clusters

// Every thread of every CTA of the cluster arrives, then waits (release /
// acquire: shared-memory writes before it are visible to the cluster after it).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// A float in the shared memory of the cluster's CTA `rank`, at the address
// that `p` has in this CTA.
__device__ __forceinline__ float ld_dsmem_f32(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
  return v;
}

__device__ __forceinline__ float block_max(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float t = lane < nw ? scratch[lane] : 0.f;
  return warp_max(t);
}

__device__ __forceinline__ float block_sum(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float t = lane < nw ? scratch[lane] : 0.f;
  return warp_sum(t);
}

}  // namespace mbt
