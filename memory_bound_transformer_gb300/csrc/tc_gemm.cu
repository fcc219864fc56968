// Host side of the tensor-core GEMMs (tc_stream.cu): the tensor-map encoder
// (looked up once through the runtime's driver entry point), the maps over
// weights and 16-bit activation rows, and the fp32 <-> high/low row kernels the
// kernel-level entry points use around a projection.
#include <algorithm>

#include "tcgen05.cuh"

namespace mbt {

constexpr int kFromHlChunk = 1024;                 // values of a row per CTA in the two kernels below

// fp32 rows -> 16-bit (BF16, or FP16 when f16) high/low rows [2 * Rp][K] (rows B..Rp-1 zero),
// a row spread over blockIdx.y chunks of 1024 values.
__global__ void to_hl_kernel(const float* x, int B, int Rp, int K, uint16_t* hl, int f16) {
  const int b = blockIdx.x;
  const int k1 = min(K, (int)(blockIdx.y + 1) * kFromHlChunk);
  for (int k = blockIdx.y * kFromHlChunk + threadIdx.x; k < k1; k += blockDim.x) {
    const float v = b < B ? x[(size_t)b * K + k] : 0.f;
    store_hl16(hl + (size_t)b * K + k, hl + (size_t)(Rp + b) * K + k, v, f16);
  }
}

__device__ __forceinline__ float hl16_to_f32(uint16_t u, int f16) {
  return f16 ? __half2float(__ushort_as_half(u)) : __uint_as_float((uint32_t)u << 16);
}

// act[b][j] = hi + lo of the SwiGLU epilogue's high/low rows; a row is spread
// over blockIdx.y chunks of 1024 values (one CTA per row left most SMs idle).
__global__ void from_hl_kernel(const uint16_t* hl, int B, int Rp, int N, float* out, int f16) {
  const int b = blockIdx.x;
  const int j1 = min(N, (int)(blockIdx.y + 1) * kFromHlChunk);
  for (int j = blockIdx.y * kFromHlChunk + threadIdx.x; j < j1; j += blockDim.x)
    out[(size_t)b * N + j] = hl16_to_f32(hl[(size_t)b * N + j], f16) + hl16_to_f32(hl[(size_t)(Rp + b) * N + j], f16);
}

// Rows (fp32 x, or 16-bit high/low rows hl [2 * Rp][K]) -> four e4m3 term rows
// t [4][Rp][K] and the rows' power-of-two scales ts[Rp] (split_terms); rows
// B..Rp-1 get zero codes and scale 1. A row is spread over a cluster of C CTAs
// that hold their slices in registers and exchange their largest |x| through
// distributed shared memory, so the row is read once.
constexpr int kTermThreads = 256;
constexpr int kTermG = 4;          // float4 per thread: K <= 8 CTAs x 256 threads x 4 x 4
__global__ void __launch_bounds__(kTermThreads) to_terms_kernel(const float* x, const uint16_t* hl, int f16, int B,
                                                                int Rp, int K, uint8_t* t, float* ts) {
  __shared__ float scratch[32];
  __shared__ float part;
  const int C = gridDim.x, c = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  const int n4 = K / 4, per = (n4 + C - 1) / C, i0 = c * per, i1 = min(n4, i0 + per);
  if (b >= B) {                    // padding rows (the whole cluster)
    for (int tj = 0; tj < kTerms; ++tj)
      for (int i = i0 + tid; i < i1; i += kTermThreads)
        reinterpret_cast<uint32_t*>(t + ((size_t)tj * Rp + b) * K)[i] = 0u;
    if (c == 0 && tid == 0) ts[b] = 1.f;
    return;
  }
  float v[kTermG][4];
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < kTermG; ++j) {
    const int i = i0 + tid + j * kTermThreads;
    if (i < i1) {
      if (x) {
        const float4 q = reinterpret_cast<const float4*>(x + (size_t)b * K)[i];
        v[j][0] = q.x; v[j][1] = q.y; v[j][2] = q.z; v[j][3] = q.w;
      } else {
        const uint2 h = reinterpret_cast<const uint2*>(hl + (size_t)b * K)[i];
        const uint2 l = reinterpret_cast<const uint2*>(hl + (size_t)(Rp + b) * K)[i];
        const uint32_t hw[4] = {h.x & 0xffffu, h.x >> 16, h.y & 0xffffu, h.y >> 16};
        const uint32_t lw[4] = {l.x & 0xffffu, l.x >> 16, l.y & 0xffffu, l.y >> 16};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          v[j][e] = f16 ? __half2float(__ushort_as_half((uint16_t)hw[e])) + __half2float(__ushort_as_half((uint16_t)lw[e]))
                        : __uint_as_float(hw[e] << 16) + __uint_as_float(lw[e] << 16);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) m = fmaxf(m, fabsf(v[j][e]));
    }
  }
  m = block_max(m, scratch);
  if (C > 1) {
    if (tid == 0) part = m;
    cluster_sync_all();
    m = 0.f;
    for (int q = 0; q < C; ++q) m = fmaxf(m, ld_dsmem_f32(&part, (uint32_t)q));
  }
  float sc, isc;
  term_scale(m, sc, isc);
  if (c == 0 && tid == 0) ts[b] = sc;
#pragma unroll
  for (int j = 0; j < kTermG; ++j) {
    const int i = i0 + tid + j * kTermThreads;
    if (i < i1) {
      uint32_t cd[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) cd[e] = split_terms(v[j][e], isc);
#pragma unroll
      for (int tj = 0; tj < kTerms; ++tj) {
        const uint32_t w = ((cd[0] >> (8 * tj)) & 255u) | (((cd[1] >> (8 * tj)) & 255u) << 8) |
                           (((cd[2] >> (8 * tj)) & 255u) << 16) | (((cd[3] >> (8 * tj)) & 255u) << 24);
        reinterpret_cast<uint32_t*>(t + ((size_t)tj * Rp + b) * K)[i] = w;
      }
    }
  }
  if (C > 1) cluster_sync_all();   // no CTA leaves while the others may still read its maximum
}

cudaError_t tc_to_terms(const float* x, const bf16* hl, int f16, int B, int Rp, int K, uint8_t* t, float* ts,
                        cudaStream_t s) {
  const int n4 = K / 4;
  const int C = std::min(8, (n4 + kTermThreads - 1) / kTermThreads);
  if (K % 4 || K < 4 || (!x && !hl) || B < 0 || B > Rp || (n4 + C - 1) / C > kTermThreads * kTermG)
    return cudaErrorInvalidValue;
  const uint16_t* h16 = reinterpret_cast<const uint16_t*>(hl);
  void* p[] = {&x, &h16, &f16, &B, &Rp, &K, &t, &ts};
  return launch_ex((const void*)to_terms_kernel, dim3(C, Rp), dim3(kTermThreads), 0, s, p, true, -1, C > 1 ? C : 0);
}

cudaError_t tc_to_hl(const float* x, int B, int Rp, int K, bf16* hl, cudaStream_t s, int f16) {
  to_hl_kernel<<<dim3(Rp, (K + kFromHlChunk - 1) / kFromHlChunk), 256, 0, s>>>(x, B, Rp, K,
                                                                               reinterpret_cast<uint16_t*>(hl), f16);
  return cudaGetLastError();
}
cudaError_t tc_from_hl(const bf16* hl, int B, int Rp, int N, float* out, cudaStream_t s, int f16) {
  from_hl_kernel<<<dim3(B, (N + kFromHlChunk - 1) / kFromHlChunk), 256, 0, s>>>(reinterpret_cast<const uint16_t*>(hl), B,
                                                                              Rp, N, out, f16);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// host side

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

}  // namespace

cudaError_t tc_init() {
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = (EncodeTiledFn)fn;
  }
  return ts_init();
}

// 2-D BF16 tensor map over [rows][K] (K contiguous), box of 64 K-elements x
// box_rows rows, 128-byte swizzle, zero fill out of bounds.
cudaError_t tc_make_map(void* map, const void* base, int rows, int K, int box_rows) {
  if (!g_encode) return cudaErrorNotSupported;
  if (((uintptr_t)base & 15) || (K * 2) % 16 || box_rows < 1 || box_rows > 256) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTcBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode((CUtensorMap*)map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2-D tensor map over e4m3 codes [rows][K] (K contiguous: weights, or the
// activations' term rows), box of 128 codes x box_rows rows, 128-byte swizzle
// (the layout the MMA's shared-memory descriptors read), zero fill out of bounds.
cudaError_t tc_make_map_u8(void* map, const void* base, int rows, int K, int box_rows) {
  if (!g_encode) return cudaErrorNotSupported;
  if (((uintptr_t)base & 15) || K % 16 || box_rows < 1 || box_rows > 256) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode((CUtensorMap*)map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace mbt
