// Host side of the tensor-core GEMMs (tc_stream.cu): the tensor-map encoder
// (looked up once through the runtime's driver entry point), the maps over
// weights and 16-bit activation rows, and the fp32 <-> high/low row kernels the
// kernel-level entry points use around a projection.
#include "tcgen05.cuh"

namespace mbt {

// fp32 rows -> 16-bit (BF16, or FP16 when f16) high/low rows [2 * Rp][K] (rows B..Rp-1 zero).
__global__ void to_hl_kernel(const float* x, int B, int Rp, int K, uint16_t* hl, int f16) {
  const int b = blockIdx.x;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const float v = b < B ? x[(size_t)b * K + k] : 0.f;
    store_hl16(hl + (size_t)b * K + k, hl + (size_t)(Rp + b) * K + k, v, f16);
  }
}

__device__ __forceinline__ float hl16_to_f32(uint16_t u, int f16) {
  return f16 ? __half2float(__ushort_as_half(u)) : __uint_as_float((uint32_t)u << 16);
}

// act[b][j] = hi + lo of the SwiGLU epilogue's high/low rows.
__global__ void from_hl_kernel(const uint16_t* hl, int B, int Rp, int N, float* out, int f16) {
  const int b = blockIdx.x;
  for (int j = threadIdx.x; j < N; j += blockDim.x)
    out[(size_t)b * N + j] = hl16_to_f32(hl[(size_t)b * N + j], f16) + hl16_to_f32(hl[(size_t)(Rp + b) * N + j], f16);
}

cudaError_t tc_to_hl(const float* x, int B, int Rp, int K, bf16* hl, cudaStream_t s, int f16) {
  to_hl_kernel<<<Rp, 256, 0, s>>>(x, B, Rp, K, reinterpret_cast<uint16_t*>(hl), f16);
  return cudaGetLastError();
}
cudaError_t tc_from_hl(const bf16* hl, int B, int Rp, int N, float* out, cudaStream_t s, int f16) {
  from_hl_kernel<<<B, 256, 0, s>>>(reinterpret_cast<const uint16_t*>(hl), B, Rp, N, out, f16);
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

// 2-D tensor map over e4m3 codes [rows][K] (K contiguous), box of 128 codes x
// 64 rows, 128-byte swizzle (16-byte chunk c of row r lands at chunk
// c ^ (r % 8), so the widening threads, one row each, read shared memory
// without bank conflicts), zero fill out of bounds.
cudaError_t tc_make_map_u8(void* map, const void* base, int rows, int K) {
  if (!g_encode) return cudaErrorNotSupported;
  if (((uintptr_t)base & 15) || K % 16) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {128u, 64u};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode((CUtensorMap*)map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace mbt
