// Skinny GEMM on the 5th-generation tensor cores for decode at batch 16..128.
//
// At these batches a projection is a real dense contraction: the weight-only
// arithmetic intensity 2B / b_w ("GPU Inference Internals", "Roofline: Why
// Decode Is Memory-Bound") reaches 16-128 FLOP per byte, beyond what the CUDA
// cores sustain at HBM rate, so the projection runs as tcgen05 MMAs:
//   * swap-AB: the weights are the M = 128 operand (one tile = 128 output
//     channels x the K range of the CTA), the batch rows are N;
//   * the activations are fp32; each row is split into a BF16 high part and a
//     BF16 low part (x = hi + lo to ~2^-17 relative) and the two are stacked
//     along N, so one MMA with N = 2 * rows keeps near-fp32 accuracy while the
//     weights are read once;
//   * TMA moves 128-byte-swizzled K-major tiles of both operands into a
//     3-stage shared-memory ring (two CTAs per SM); one thread issues the TMA copies, one thread
//     issues the MMAs into a TMEM accumulator, mbarriers hand stages back and
//     forth (every wait is bounded: on a timeout the kernel flags the error
//     word, frees its TMEM and returns);
//   * epilogues read TMEM with tcgen05.ld: split-K partial sums, SwiGLU over a
//     tile of 64 gate + 64 up rows (written back as hi/lo BF16 for the down
//     projection), or a per-tile arg-max for the LM head.
#include "tcgen05.cuh"

namespace mbt {

constexpr int kTcThreads = 128;
#ifndef MBT_TC_STAGES
#define MBT_TC_STAGES 3
#endif
constexpr int kTcStages = MBT_TC_STAGES;   // 3 x 32 KB at 64 rows: two CTAs fit an SM
template <int EPI>
__global__ void __launch_bounds__(kTcThreads, kTcTP == 1 ? 2 : 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const TcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[kTcStages], empty[kTcStages], done;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ int have_s, issued_s, consumed_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // kTcTP weight tiles per CTA share every activation tile
  const int tile0 = blockIdx.x * kTcTP, split = blockIdx.y;
  const int ntiles = EPI == EPI_SWIGLU ? (a.N + 63) / 64 : (a.N + kTcBM - 1) / kTcBM;
  const int Rp = a.Rp, NM = 2 * Rp;                // MMA N: hi rows then lo rows
  const uint32_t at_bytes = kTcBM * 128, a_bytes = kTcTP * at_bytes, b_bytes = (uint32_t)NM * 128;
  unsigned char* sA = smem;
  unsigned char* sB = smem + kTcStages * a_bytes;
  const int nk_all = (a.K + kTcBK - 1) / kTcBK;
  const int kc0 = (int)((long long)nk_all * split / gridDim.y);
  const int nk = (int)((long long)nk_all * (split + 1) / gridDim.y) - kc0;
  // weight rows of each tile's two 64-row halves (SwiGLU: gate half, up half)
  auto rowA0 = [&](int t) { return EPI == EPI_SWIGLU ? t * 64 : t * kTcBM; };
  auto rowA1 = [&](int t) { return EPI == EPI_SWIGLU ? a.N + t * 64 : t * kTcBM + 64; };

  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    mbar_init(&done, 1);
    abort_flag = 0;
    issued_s = 0;
    consumed_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
  }
  const int ncols = kTcTP * NM;
  const uint32_t tcols = ncols <= 32 ? 32 : ncols <= 64 ? 64 : ncols <= 128 ? 128 : ncols <= 256 ? 256 : 512;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(&tmem_slot)), "r"(tcols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0 && lane == 0) {
    // producer: the weight tiles do not depend on the previous kernel, so the
    // first stages' weights are requested before waiting for it
    const int pre = nk < kTcStages ? nk : kTcStages;
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_tx(&full[i], a_bytes + b_bytes);
      const int kx = (kc0 + i) * kTcBK;
      for (int j = 0; j < kTcTP; ++j) {
        tma_load_2d(sA + i * a_bytes + j * at_bytes, &tmW, kx, rowA0(tile0 + j), &full[i]);
        tma_load_2d(sA + i * a_bytes + j * at_bytes + 64 * 128, &tmW, kx, rowA1(tile0 + j), &full[i]);
      }
    }
    pdl_wait();
    for (int i = 0; i < pre; ++i) tma_load_2d(sB + i * b_bytes, &tmX, (kc0 + i) * kTcBK, 0, &full[i]);
    int issued = pre;
    for (int i = pre; i < nk; ++i) {
      const int s = i % kTcStages;
      if (abort_flag || !mbar_wait(&empty[s], ((i / kTcStages) - 1) & 1)) { abort_flag = 1; break; }
      mbar_arrive_tx(&full[s], a_bytes + b_bytes);
      const int kx = (kc0 + i) * kTcBK;
      for (int j = 0; j < kTcTP; ++j) {
        tma_load_2d(sA + s * a_bytes + j * at_bytes, &tmW, kx, rowA0(tile0 + j), &full[s]);
        tma_load_2d(sA + s * a_bytes + j * at_bytes + 64 * 128, &tmW, kx, rowA1(tile0 + j), &full[s]);
      }
      tma_load_2d(sB + s * b_bytes, &tmX, kx, 0, &full[s]);
      issued = i + 1;
    }
    issued_s = issued;
  } else if (warp == 1 && lane == 0) {
    pdl_wait();
    // MMA issuer: 4 MMAs of K = 16 per 64-element stage
    const uint32_t idesc = idesc_16(kTcBM, NM, 0);
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int s = i % kTcStages;
      if (abort_flag || !mbar_wait(&full[s], (i / kTcStages) & 1)) { abort_flag = 1; ok = false; break; }
      consumed_s = i + 1;
      tc_fence_after();
      const uint64_t bd = sw128_desc(smem_u32(sB + s * b_bytes));
#pragma unroll
      for (int j = 0; j < kTcTP; ++j) {
        const uint64_t ad = sw128_desc(smem_u32(sA + s * a_bytes + j * at_bytes));
#pragma unroll
        for (int kk = 0; kk < kTcBK / 16; ++kk)
          umma_kf16(tmem + (uint32_t)(j * NM), ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                    (i > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(&empty[s]);
    }
    if (ok) umma_commit(&done);
    else mbar_arrive_tx(&done, 0);                // release the epilogue without MMAs
  } else {
    pdl_wait();
  }
  __syncwarp();

  // epilogue: every thread owns one TMEM lane = one weight row of the tile;
  // whether there is a result is decided once for the whole CTA
  const bool done_ok = mbar_wait(&done, 0);
  __syncthreads();
  if (tid == 0) have_s = done_ok && !abort_flag && nk > 0;
  __syncthreads();
  const bool have = have_s != 0;
  tc_fence_after();
  if (!have) {
    if (tid == 0 && (abort_flag || nk > 0)) set_err(a.err, MBT_DEV_WAIT_LIMIT);
  } else {
    for (int j = 0; j < kTcTP && tile0 + j < ntiles; ++j) {
      if (j) named_bar(1, kTcThreads);                                   // the scratch is reused
      tc_epilogue<EPI>(a, tmem + (uint32_t)(j * NM), warp, lane, tid, tile0 + j, split, sA, 1);   // ring free
    }
  }

  // teardown: no TMA or MMA of this CTA is still in flight once `done` fired;
  // after a timeout, wait (bounded) for the copies the producer issued but the
  // MMA thread never consumed before the shared memory is released
  if (abort_flag && tid == 0) {
    for (int i = consumed_s; i < issued_s; ++i) mbar_wait(&full[i % kTcStages], (i / kTcStages) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tcols) : "memory");
  }
}

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

template <int EPI>
void* tc_fn() { return (void*)tc_gemm_kernel<EPI>; }
void* tc_pick(int epi) {
  return epi == EPI_PARTIAL ? tc_fn<EPI_PARTIAL>() : epi == EPI_SWIGLU ? tc_fn<EPI_SWIGLU>() : tc_fn<EPI_ARGMAX>();
}
}  // namespace

size_t tc_smem(int Rp);

cudaError_t tc_init() {
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = (EncodeTiledFn)fn;
  }
  for (int epi = 0; epi < 3; ++epi) {
    cudaError_t e = cudaFuncSetAttribute(tc_pick(epi), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)tc_smem(128));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
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

// 2-D tensor map over e4m3 codes [rows][K] (K contiguous), box of 64 codes x
// 64 rows, 64-byte swizzle (16-byte chunk c of row r lands at chunk
// c ^ ((r / 2) % 4), so the widening threads, one row each, read shared memory
// without bank conflicts), zero fill out of bounds.
cudaError_t tc_make_map_u8(void* map, const void* base, int rows, int K) {
  if (!g_encode) return cudaErrorNotSupported;
  if (((uintptr_t)base & 15) || K % 16) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {(cuuint32_t)kTcBK, 64u};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode((CUtensorMap*)map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

size_t tc_smem(int Rp) { return 1024 + (size_t)kTcStages * (kTcTP * kTcBM * 128 + (size_t)2 * Rp * 128); }

int tc_tiles(int epi, int N) { return epi == EPI_SWIGLU ? (N + 63) / 64 : (N + kTcBM - 1) / kTcBM; }

cudaError_t tc_launch(int epi, const void* mapW, const void* mapX, const TcArgs& a, int ksplit, cudaStream_t s) {
  CUtensorMap w = *(const CUtensorMap*)mapW, x = *(const CUtensorMap*)mapX;
  TcArgs args = a;
  void* params[] = {&w, &x, &args};
  return launch_pdl(tc_pick(epi), dim3((tc_tiles(epi, a.N) + kTcTP - 1) / kTcTP, ksplit), dim3(kTcThreads),
                    tc_smem(a.Rp), s, params);
}

}  // namespace mbt
