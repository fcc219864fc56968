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
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace mbt {

constexpr int kTcThreads = 128;
constexpr int kTcBM = 128;              // weight rows per tile (MMA M)
constexpr int kTcBK = 64;               // K elements per stage: one 128-byte swizzle row of BF16
constexpr int kTcStages = 3;            // 3 x 32 KB at 64 rows: two CTAs fit an SM
constexpr long long kTcWaitCycles = 4000000000LL;   // about 2 s at GB300 clocks

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(b)), "r"(parity) : "memory");
  return ok != 0;
}
// Wait for a phase; false once the time limit has passed.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
  if (mbar_try(b, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try(b, parity))
    if (clock64() - t0 > kTcWaitCycles) return false;
  return true;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar)) : "memory");
}

// Shared-memory matrix descriptor: K-major tile of 128-byte rows, 128-byte
// swizzle, 8-row (1024-byte) atoms stacked along M/N.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);        // start address
  d |= (uint64_t)1 << 16;                         // leading byte offset (unused here), 16 B
  d |= (uint64_t)(1024 >> 4) << 32;               // stride byte offset: one 8-row atom
  d |= (uint64_t)1 << 46;                         // descriptor version
  d |= (uint64_t)2 << 61;                         // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: BF16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 8 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

template <int EPI>
__global__ void __launch_bounds__(kTcThreads, 2)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const TcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[kTcStages], empty[kTcStages], done;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ int have_s, issued_s, consumed_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int Rp = a.Rp, NM = 2 * Rp;                // MMA N: hi rows then lo rows
  const uint32_t a_bytes = kTcBM * 128, b_bytes = (uint32_t)NM * 128;
  unsigned char* sA = smem;
  unsigned char* sB = smem + kTcStages * a_bytes;
  const int nk_all = (a.K + kTcBK - 1) / kTcBK;
  const int kc0 = (int)((long long)nk_all * split / gridDim.y);
  const int nk = (int)((long long)nk_all * (split + 1) / gridDim.y) - kc0;
  // weight rows of the tile's two 64-row halves (SwiGLU: gate half, up half)
  const int rowA0 = EPI == EPI_SWIGLU ? tile * 64 : tile * kTcBM;
  const int rowA1 = EPI == EPI_SWIGLU ? a.N + tile * 64 : tile * kTcBM + 64;

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
  const uint32_t tcols = NM <= 32 ? 32 : NM <= 64 ? 64 : NM <= 128 ? 128 : 256;
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
      tma_load_2d(sA + i * a_bytes, &tmW, kx, rowA0, &full[i]);
      tma_load_2d(sA + i * a_bytes + 64 * 128, &tmW, kx, rowA1, &full[i]);
    }
    pdl_wait();
    for (int i = 0; i < pre; ++i) tma_load_2d(sB + i * b_bytes, &tmX, (kc0 + i) * kTcBK, 0, &full[i]);
    int issued = pre;
    for (int i = pre; i < nk; ++i) {
      const int s = i % kTcStages;
      if (abort_flag || !mbar_wait(&empty[s], ((i / kTcStages) - 1) & 1)) { abort_flag = 1; break; }
      mbar_arrive_tx(&full[s], a_bytes + b_bytes);
      const int kx = (kc0 + i) * kTcBK;
      tma_load_2d(sA + s * a_bytes, &tmW, kx, rowA0, &full[s]);
      tma_load_2d(sA + s * a_bytes + 64 * 128, &tmW, kx, rowA1, &full[s]);
      tma_load_2d(sB + s * b_bytes, &tmX, kx, 0, &full[s]);
      issued = i + 1;
    }
    issued_s = issued;
  } else if (warp == 1 && lane == 0) {
    pdl_wait();
    // MMA issuer: 4 MMAs of K = 16 per 64-element stage
    const uint32_t idesc = idesc_bf16(kTcBM, NM);
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int s = i % kTcStages;
      if (abort_flag || !mbar_wait(&full[s], (i / kTcStages) & 1)) { abort_flag = 1; ok = false; break; }
      consumed_s = i + 1;
      tc_fence_after();
      const uint64_t ad = sw128_desc(smem_u32(sA + s * a_bytes));
      const uint64_t bd = sw128_desc(smem_u32(sB + s * b_bytes));
#pragma unroll
      for (int kk = 0; kk < kTcBK / 16; ++kk)
        umma_bf16(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (i > 0 || kk > 0) ? 1u : 0u);
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
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  const int row = warp * 32 + lane;
  if (!have) {
    if (tid == 0 && (abort_flag || nk > 0)) set_err(a.err, MBT_DEV_WAIT_LIMIT);
  } else if (EPI == EPI_PARTIAL) {
    const int n = tile * kTcBM + row;
    const float sc = (a.scale && n < a.N) ? a.scale[n] : 1.f;
    for (int c0 = 0; c0 < Rp; c0 += 8) {
      float hi[8], lo[8];
      tmem_ld8(lane_base + c0, hi);
      tmem_ld8(lane_base + Rp + c0, lo);
      if (n < a.N) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (c0 + j < a.R)
            a.out[(size_t)split * a.split_stride + (size_t)(c0 + j) * a.ldo + n] = (hi[j] + lo[j]) * sc;
      }
    }
  } else if (EPI == EPI_SWIGLU) {
    // lanes 0..63: gate rows, 64..127: up rows of channels tile*64 + (row % 64)
    float* ex = reinterpret_cast<float*>(sA);      // [64][Rp] up values (the stage ring is free now)
    const int j = tile * 64 + (row & 63);
    const bool ch_ok = j < a.N;
    if (warp >= 2) {
      const float su = (a.scale && ch_ok) ? a.scale[a.N + j] : 1.f;
      for (int c0 = 0; c0 < Rp; c0 += 8) {
        float hi[8], lo[8];
        tmem_ld8(lane_base + c0, hi);
        tmem_ld8(lane_base + Rp + c0, lo);
#pragma unroll
        for (int q = 0; q < 8; ++q) ex[(row - 64) * Rp + c0 + q] = (hi[q] + lo[q]) * su;
      }
    }
    __syncthreads();
    if (warp < 2) {
      const float sg = (a.scale && ch_ok) ? a.scale[j] : 1.f;
      for (int c0 = 0; c0 < Rp; c0 += 8) {
        float hi[8], lo[8];
        tmem_ld8(lane_base + c0, hi);
        tmem_ld8(lane_base + Rp + c0, lo);
        if (ch_ok) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int b = c0 + q;
            const float g = (hi[q] + lo[q]) * sg;
            const float u = ex[row * Rp + b];
            const float act = b < a.R ? g / (1.f + expf(-g)) * u : 0.f;
            const bf16 h = __float2bfloat16_rn(act);
            a.act_hl[(size_t)b * a.ld_act + j] = h;
            a.act_hl[(size_t)(Rp + b) * a.ld_act + j] = __float2bfloat16_rn(act - __bfloat162float(h));
          }
        }
      }
    }
  } else {  // EPI_ARGMAX
    float* bv = reinterpret_cast<float*>(sA);        // [4 warps][Rp]
    int* bi = reinterpret_cast<int*>(sA + 4 * Rp * 4);
    const int n = tile * kTcBM + row;
    const float sc = (a.scale && n < a.N) ? a.scale[n] : 1.f;
    for (int c0 = 0; c0 < Rp; c0 += 8) {
      float hi[8], lo[8];
      tmem_ld8(lane_base + c0, hi);
      tmem_ld8(lane_base + Rp + c0, lo);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int b = c0 + q;
        float v = n < a.N ? (hi[q] + lo[q]) * sc : -INFINITY;
        if (!(v == v)) { set_err(a.err, MBT_DEV_NONFINITE); v = -INFINITY; }
        if (n < a.N && b < a.R && a.logits) a.logits[(size_t)b * a.ldl + n] = v;
        int idx = n;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, v, o);
          const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
          if (ov > v || (ov == v && oi < idx)) { v = ov; idx = oi; }
        }
        if (lane == 0) { bv[warp * Rp + b] = v; bi[warp * Rp + b] = idx; }
      }
    }
    __syncthreads();
    for (int b = tid; b < a.R; b += kTcThreads) {
      float v = bv[b];
      int idx = bi[b];
      for (int w2 = 1; w2 < 4; ++w2) {
        const float ov = bv[w2 * Rp + b];
        const int oi = bi[w2 * Rp + b];
        if (ov > v || (ov == v && oi < idx)) { v = ov; idx = oi; }
      }
      ArgmaxPart p;
      p.v = v; p.i = idx;
      a.part[(size_t)tile * a.part_ld + b] = p;
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

// fp32 rows -> BF16 high/low rows [2 * Rp][K] (rows B..Rp-1 zero).
__global__ void to_hl_kernel(const float* x, int B, int Rp, int K, bf16* hl) {
  const int b = blockIdx.x;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const float v = b < B ? x[(size_t)b * K + k] : 0.f;
    const bf16 h = __float2bfloat16_rn(v);
    hl[(size_t)b * K + k] = h;
    hl[(size_t)(Rp + b) * K + k] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

// act[b][j] = hi + lo of the SwiGLU epilogue's high/low rows.
__global__ void from_hl_kernel(const bf16* hl, int B, int Rp, int N, float* out) {
  const int b = blockIdx.x;
  for (int j = threadIdx.x; j < N; j += blockDim.x)
    out[(size_t)b * N + j] = __bfloat162float(hl[(size_t)b * N + j]) + __bfloat162float(hl[(size_t)(Rp + b) * N + j]);
}

cudaError_t tc_to_hl(const float* x, int B, int Rp, int K, bf16* hl, cudaStream_t s) {
  to_hl_kernel<<<Rp, 256, 0, s>>>(x, B, Rp, K, hl);
  return cudaGetLastError();
}
cudaError_t tc_from_hl(const bf16* hl, int B, int Rp, int N, float* out, cudaStream_t s) {
  from_hl_kernel<<<B, 256, 0, s>>>(hl, B, Rp, N, out);
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

size_t tc_smem(int Rp) { return 1024 + (size_t)kTcStages * (kTcBM * 128 + (size_t)2 * Rp * 128); }

int tc_tiles(int epi, int N) { return epi == EPI_SWIGLU ? (N + 63) / 64 : (N + kTcBM - 1) / kTcBM; }

cudaError_t tc_launch(int epi, const void* mapW, const void* mapX, const TcArgs& a, int ksplit, cudaStream_t s) {
  CUtensorMap w = *(const CUtensorMap*)mapW, x = *(const CUtensorMap*)mapX;
  TcArgs args = a;
  void* params[] = {&w, &x, &args};
  return launch_pdl(tc_pick(epi), dim3(tc_tiles(epi, a.N), ksplit), dim3(kTcThreads), tc_smem(a.Rp), s, params);
}

}  // namespace mbt
