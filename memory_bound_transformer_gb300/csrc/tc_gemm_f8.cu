// Skinny GEMM on the tcgen05 tensor cores for e4m3 weights, batch 16..128.
//
// Same contraction as the BF16 skinny GEMM (swap-AB: weight rows are the
// M = 128 operand, the activation rows the N operand as 16-bit high/low
// parts), with the weights read once as e4m3 codes: "FP8 weights ... halve the
// bytes moved per step" ("Kernel Fusion for Large-Scale LLM Inference",
// section 11). kind::f16 takes two 16-bit operands of one type, so the codes
// are widened to FP16 on the way to the tensor core and the activations are
// FP16 high/low rows; the per-row scale is applied in the epilogue ("Epilogue
// and dequant fusion", same section).
//
// Where the widened weights live decides the speed. An MMA of M = 128, N = 128
// reading both operands from shared memory already takes its full bandwidth,
// so a widened FP16 tile written to and read back from shared memory (on top
// of the raw codes and the activations) leaves the stage bound by shared
// memory, not HBM. Here the widening warps put the FP16 weights into tensor
// memory and the MMA reads A from there (tcgen05.mma with A in TMEM); shared
// memory carries only the raw codes (written by TMA, read once by the
// widening threads) and the activation tiles.
//
// Widening without a conversion instruction: an e4m3 code s.eeee.mmm has
// value (-1)^s 2^(e-7) (1 + m/8) (subnormal at e = 0: 2^-6 m/8). The FP16
// pattern s.0eeee.mmm0000000 has value (-1)^s 2^(e-15) (1 + m/8) (subnormal at
// e = 0: 2^-14 m/8), i.e. exactly the e4m3 value / 256 for every finite code,
// subnormals included. So each code pair becomes one FP16x2 word with a byte
// permute, a shift and masks, and the factor 256 joins the per-row scale in the
// epilogue (a power of two: no rounding). The two NaN codes (S.1111.111) are
// not valid weights: they widen to +-480 instead of NaN.
//
// Warp roles (256 threads):
//   warp 0 (one thread): TMA copies of raw 64-code x 128-row tiles (8 KB,
//                        64-byte swizzle) into a ring: the bytes in flight
//                        that keep HBM busy; it never waits on the previous
//                        kernel (the weights do not depend on it);
//   warp 1 (one thread): TMA copies of the activation tiles;
//   warp 2 (one thread): the MMAs (A from TMEM, B from shared memory) and
//                        their commits;
//   warps 4-7:           warp 4 + q owns TMEM lanes 32q..32q+31 = weight rows
//                        32q..32q+31 of the tile: each thread widens its row's
//                        64 codes per stage into one 32-column A stage of
//                        TMEM, and the same warps run the epilogue.
// Every wait is bounded (about 2 s): on a timeout the kernel flags
// MBT_DEV_WAIT_LIMIT, lets its issued MMAs and copies finish (bounded), frees
// its TMEM and returns.
#include "tcgen05.cuh"

namespace mbt {

#ifndef MBT_F8_RAW
#define MBT_F8_RAW 10
#endif
#ifndef MBT_F8_ASTAGES
#define MBT_F8_ASTAGES 6
#endif
#ifndef MBT_F8_BST
#define MBT_F8_BST 4
#endif
constexpr int kF8Threads = 256;
constexpr int kF8Raw = MBT_F8_RAW;                // raw e4m3 stages in shared memory
constexpr int kF8A = MBT_F8_ASTAGES;              // widened A stages in TMEM
constexpr int kF8B = MBT_F8_BST;                  // activation stages
constexpr uint32_t kF8RawBytes = kTcBM * kTcBK;   // 128 rows x 64 codes
constexpr uint32_t kF8AccCols = 256;              // accumulator: 2 * Rp <= 256 fp32 columns
constexpr uint32_t kF8ACols = kTcBK / 2;          // one A stage: 64 FP16 per row = 32 columns
constexpr uint32_t kF8TmemCols = 512;
static_assert(kF8AccCols + kF8A * kF8ACols <= kF8TmemCols, "TMEM budget");
constexpr float kF8Widen = 256.f;                 // FP16 pattern value x 256 = e4m3 value

// Dynamic shared memory of one CTA: at least 120 KB, so that two CTAs never
// share an SM (each takes all 512 TMEM columns).
size_t tc8_smem(int Rp) {
  const size_t need = 1024 + (size_t)kF8Raw * kF8RawBytes + (size_t)kF8B * 2 * Rp * 128;
  return need > (size_t)120 * 1024 ? need : (size_t)120 * 1024;
}

// Four e4m3 codes (a 32-bit word, lowest byte first) -> two FP16x2 words of
// value / 256 (see the file comment).
__device__ __forceinline__ void widen4_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t t0 = __byte_perm(w, 0u, 0x1404);   // code 0 in byte 1, code 1 in byte 3
  const uint32_t t1 = __byte_perm(w, 0u, 0x3424);   // code 2 in byte 1, code 3 in byte 3
  lo = ((t0 >> 1) & 0x3F803F80u) | (t0 & 0x80008000u);
  hi = ((t1 >> 1) & 0x3F803F80u) | (t1 & 0x80008000u);
}

template <int EPI>
__global__ void __launch_bounds__(kF8Threads, 1)
tc_gemm_f8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const TcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t raw_full[kF8Raw], raw_empty[kF8Raw], a_full[kF8A], a_empty[kF8A];
  __shared__ __align__(8) uint64_t b_full[kF8B], b_empty[kF8B], done;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ int have_s, raw_issued_s, raw_used_s, b_issued_s, b_used_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int Rp = a.Rp, NM = 2 * Rp;
  const uint32_t b_bytes = (uint32_t)NM * 128;
  unsigned char* sR = smem;                                           // [kF8Raw][128 rows][64 B], 64-B swizzle
  unsigned char* sB = sR + kF8Raw * kF8RawBytes;                      // [kF8B][NM rows][128 B], 128-B swizzle
  const int nk_all = (a.K + kTcBK - 1) / kTcBK;
  const int kc0 = (int)((long long)nk_all * split / gridDim.y);
  const int nk = (int)((long long)nk_all * (split + 1) / gridDim.y) - kc0;
  const int rowA0 = EPI == EPI_SWIGLU ? tile * 64 : tile * kTcBM;
  const int rowA1 = EPI == EPI_SWIGLU ? a.N + tile * 64 : tile * kTcBM + 64;

  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < kF8Raw; ++s) { mbar_init(&raw_full[s], 1); mbar_init(&raw_empty[s], 4); }
    for (int s = 0; s < kF8A; ++s) { mbar_init(&a_full[s], 4); mbar_init(&a_empty[s], 1); }
    for (int s = 0; s < kF8B; ++s) { mbar_init(&b_full[s], 1); mbar_init(&b_empty[s], 1); }
    mbar_init(&done, 1);
    abort_flag = 0;
    raw_issued_s = raw_used_s = b_issued_s = b_used_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(&tmem_slot)), "r"(kF8TmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;                    // accumulator at columns [0, NM)
  const uint32_t tmem_a = tmem + kF8AccCols;          // A stage j at columns kF8AccCols + 32 j

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % kF8Raw;
        if (i >= kF8Raw && (abort_flag || !mbar_wait(&raw_empty[s], ((i / kF8Raw) - 1) & 1))) { abort_flag = 1; break; }
        mbar_arrive_tx(&raw_full[s], kF8RawBytes);
        const int kx = (kc0 + i) * kTcBK;
        tma_load_2d(sR + s * kF8RawBytes, &tmW, kx, rowA0, &raw_full[s]);
        tma_load_2d(sR + s * kF8RawBytes + 64 * kTcBK, &tmW, kx, rowA1, &raw_full[s]);
        issued = i + 1;
      }
      raw_issued_s = issued;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      pdl_wait();
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % kF8B;
        if (i >= kF8B && (abort_flag || !mbar_wait(&b_empty[s], ((i / kF8B) - 1) & 1))) { abort_flag = 1; break; }
        mbar_arrive_tx(&b_full[s], b_bytes);
        tma_load_2d(sB + s * b_bytes, &tmX, (kc0 + i) * kTcBK, 0, &b_full[s]);
        issued = i + 1;
      }
      b_issued_s = issued;
    }
  } else if (warp == 2) {
    if (lane == 0) {
      pdl_wait();
      const uint32_t idesc = idesc_16(kTcBM, NM, 1);
      for (int i = 0; i < nk; ++i) {
        const int j = i % kF8A, s = i % kF8B;
        if (abort_flag || !mbar_wait(&a_full[j], (i / kF8A) & 1) || !mbar_wait(&b_full[s], (i / kF8B) & 1)) {
          abort_flag = 1;
          break;
        }
        b_used_s = i + 1;
        tc_fence_after();
        const uint64_t bd = sw128_desc(smem_u32(sB + s * b_bytes));
        const uint32_t ta = tmem_a + (uint32_t)(j * kF8ACols);
#pragma unroll
        for (int kk = 0; kk < kTcBK / 16; ++kk)
          umma_kf16_tmem_a(tmem, ta + (uint32_t)(kk * 8), bd + (uint64_t)(kk * 2), idesc, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&a_empty[j]);
        umma_commit(&b_empty[s]);
      }
      // after the last MMA this CTA issued, aborted or not: `done` fires once
      // all of them have completed, so TMEM is never freed under an MMA
      umma_commit(&done);
    }
  } else if (warp >= 4) {
    // widening: thread = row q*32 + lane of the tile = TMEM lane
    const int q = warp - 4, row = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int sw = (row >> 1) & 3;                     // 64-byte swizzle of this row's 16-byte chunks
    for (int i = 0; i < nk; ++i) {
      const int r = i % kF8Raw, j = i % kF8A;
      if (abort_flag || !mbar_wait(&raw_full[r], (i / kF8Raw) & 1) ||
          (i >= kF8A && !mbar_wait(&a_empty[j], ((i / kF8A) - 1) & 1))) {
        abort_flag = 1;
        break;
      }
      const unsigned char* src = sR + r * kF8RawBytes + row * kTcBK;
      uint4 w[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint4*>(src + ((c ^ sw) * 16));
      __syncwarp();
      if (lane == 0) mbar_arrive(&raw_empty[r]);      // the codes are in registers: the slot may refill
      if (q == 0 && lane == 0) raw_used_s = i + 1;
      uint32_t h[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        widen4_f16(w[c].x, h[8 * c + 0], h[8 * c + 1]);
        widen4_f16(w[c].y, h[8 * c + 2], h[8 * c + 3]);
        widen4_f16(w[c].z, h[8 * c + 4], h[8 * c + 5]);
        widen4_f16(w[c].w, h[8 * c + 6], h[8 * c + 7]);
      }
      tmem_st32(tmem_a + lane_off + (uint32_t)(j * kF8ACols), h);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[j]);
    }
  }
  __syncwarp();

  // epilogue by warps 4..7 (TMEM lane quarter = warp % 4)
  const bool done_ok = mbar_wait(&done, 0);
  __syncthreads();
  if (tid == 0) have_s = done_ok && !abort_flag && nk > 0;
  __syncthreads();
  tc_fence_after();
  if (warp >= 4) {
    if (!have_s) {
      if (tid == 128 && (abort_flag || nk > 0)) set_err(a.err, MBT_DEV_WAIT_LIMIT);
    } else {
      tc_epilogue<EPI>(a, tmem, warp & 3, lane, tid - 128, tile, split, sR, 1, kF8Widen);   // the raw ring is free now
    }
  }

  // teardown: `done` covers every MMA; after a timeout, wait (bounded) for
  // copies that were issued and never consumed before shared memory is released
  if (abort_flag && tid == 0) {
    for (int i = raw_used_s; i < raw_issued_s; ++i) mbar_wait(&raw_full[i % kF8Raw], (i / kF8Raw) & 1);
    for (int i = b_used_s; i < b_issued_s; ++i) mbar_wait(&b_full[i % kF8B], (i / kF8B) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kF8TmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// host side

namespace {
template <int EPI>
void* tc8_fn() { return (void*)tc_gemm_f8_kernel<EPI>; }
void* tc8_pick(int epi) {
  return epi == EPI_PARTIAL ? tc8_fn<EPI_PARTIAL>() : epi == EPI_SWIGLU ? tc8_fn<EPI_SWIGLU>() : tc8_fn<EPI_ARGMAX>();
}
}  // namespace

cudaError_t tc8_init() {
  for (int epi = 0; epi < 3; ++epi) {
    cudaError_t e = cudaFuncSetAttribute(tc8_pick(epi), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)tc8_smem(128));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t tc8_launch(int epi, const void* mapW, const void* mapX, const TcArgs& a, int ksplit, cudaStream_t s) {
  CUtensorMap w = *(const CUtensorMap*)mapW, x = *(const CUtensorMap*)mapX;
  TcArgs args = a;
  void* params[] = {&w, &x, &args};
  return launch_pdl(tc8_pick(epi), dim3(tc_tiles(epi, a.N), ksplit), dim3(kF8Threads), tc8_smem(a.Rp), s, params);
}

}  // namespace mbt
