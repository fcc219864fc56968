// Skinny GEMM on the tcgen05 tensor cores for e4m3 weights, batch 16..128.
//
// Same contraction as the BF16 skinny GEMM (swap-AB: weight rows are the
// M = 128 operand, the activation rows the N operand as 16-bit high/low
// parts), with the weights read once as e4m3 codes: "FP8 weights ... halve the
// bytes moved per step" ("Kernel Fusion for Large-Scale LLM Inference",
// section 11). The MMA takes 16-bit operands of one type, so the codes are
// widened to FP16 in shared memory (exactly: every e4m3 value is an FP16
// value) between the copy engine and the tensor core, and the activations
// are FP16 high/low rows; the per-row scale is applied in the epilogue
// ("Epilogue and dequant fusion", same section). Warp roles:
//   warp 0 (one thread): TMA copies of raw e4m3 tiles into an 8-stage ring
//                        (8 KB each: the bytes in flight that keep HBM busy);
//   warp 1 (one thread): the MMAs and their commits;
//   warp 2 (one thread): TMA copies of the activation tiles (3 stages);
//   warps 3-10:          widen each raw tile into a 4-stage ring of FP16
//                        tiles in the 128-byte-swizzled K-major layout the
//                        MMA reads; warps 3-6 then run the epilogue.
// Every wait is bounded (about 2 s): on a timeout the kernel flags
// MBT_DEV_WAIT_LIMIT, waits (bounded) for the copies it issued, frees its TMEM
// and returns.
#include "tcgen05.cuh"

namespace mbt {

#ifndef MBT_F8_RAW
#define MBT_F8_RAW 8
#endif
#ifndef MBT_F8_HALF
#define MBT_F8_HALF 4
#endif
#ifndef MBT_F8_BST
#define MBT_F8_BST 3
#endif
#ifndef MBT_F8_CONV_WARPS
#define MBT_F8_CONV_WARPS 8
#endif
constexpr int kF8Conv = MBT_F8_CONV_WARPS * 32;   // widening threads (warps 3..); the first 128 run the epilogue
constexpr int kF8Threads = 96 + kF8Conv;
constexpr int kF8Items = kTcBM * 4 / kF8Conv;     // (row, 16 codes) items per widening thread per stage
constexpr int kF8Raw = MBT_F8_RAW;                // raw e4m3 stages
constexpr int kF8Half = MBT_F8_HALF;              // FP16 A stages
constexpr int kF8B = MBT_F8_BST;                  // activation stages
constexpr uint32_t kF8RawBytes = kTcBM * kTcBK;   // 128 rows x 64 codes
constexpr uint32_t kF8HalfBytes = kTcBM * 128;    // 128 rows x 64 FP16

size_t tc8_smem(int Rp) {
  return 1024 + (size_t)kF8Half * kF8HalfBytes + (size_t)kF8B * 2 * Rp * 128 + (size_t)kF8Raw * kF8RawBytes;
}

template <int EPI>
__global__ void __launch_bounds__(kF8Threads, 1)
tc_gemm_f8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const TcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t raw_full[kF8Raw], raw_empty[kF8Raw], half_full[kF8Half], half_empty[kF8Half];
  __shared__ __align__(8) uint64_t b_full[kF8B], b_empty[kF8B], done;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ int have_s, raw_issued_s, raw_used_s, b_issued_s, b_used_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int Rp = a.Rp, NM = 2 * Rp;
  const uint32_t b_bytes = (uint32_t)NM * 128;
  unsigned char* sH = smem;                                           // [kF8Half][128 rows][128 B], swizzled
  unsigned char* sB = sH + kF8Half * kF8HalfBytes;                    // [kF8B][NM rows][128 B], swizzled
  unsigned char* sR = sB + kF8B * b_bytes;                            // [kF8Raw][128 rows][64 B]
  const int nk_all = (a.K + kTcBK - 1) / kTcBK;
  const int kc0 = (int)((long long)nk_all * split / gridDim.y);
  const int nk = (int)((long long)nk_all * (split + 1) / gridDim.y) - kc0;
  const int rowA0 = EPI == EPI_SWIGLU ? tile * 64 : tile * kTcBM;
  const int rowA1 = EPI == EPI_SWIGLU ? a.N + tile * 64 : tile * kTcBM + 64;

  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < kF8Raw; ++s) { mbar_init(&raw_full[s], 1); mbar_init(&raw_empty[s], kF8Conv); }
    for (int s = 0; s < kF8Half; ++s) { mbar_init(&half_full[s], kF8Conv); mbar_init(&half_empty[s], 1); }
    for (int s = 0; s < kF8B; ++s) { mbar_init(&b_full[s], 1); mbar_init(&b_empty[s], 1); }
    mbar_init(&done, 1);
    abort_flag = 0;
    raw_issued_s = raw_used_s = b_issued_s = b_used_s = 0;
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

  if (warp == 0) {
    if (lane == 0) {
      // raw weight tiles: they do not depend on the previous kernel, so this
      // thread never waits for it
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
  } else if (warp == 2) {
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
  } else if (warp == 1) {
    if (lane == 0) {
      pdl_wait();
      const uint32_t idesc = idesc_16(kTcBM, NM, 1);
      bool ok = true;
      for (int i = 0; i < nk; ++i) {
        const int h = i % kF8Half, s = i % kF8B;
        if (abort_flag || !mbar_wait(&half_full[h], (i / kF8Half) & 1) || !mbar_wait(&b_full[s], (i / kF8B) & 1)) {
          abort_flag = 1;
          ok = false;
          break;
        }
        b_used_s = i + 1;
        tc_fence_after();
        const uint64_t ad = sw128_desc(smem_u32(sH + h * kF8HalfBytes));
        const uint64_t bd = sw128_desc(smem_u32(sB + s * b_bytes));
#pragma unroll
        for (int kk = 0; kk < kTcBK / 16; ++kk)
          umma_kf16(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&half_empty[h]);
        umma_commit(&b_empty[s]);
      }
      if (ok) umma_commit(&done);
      else mbar_arrive_tx(&done, 0);
    }
  } else {
    // warps 3..6: widen raw tile i into FP16 stage i % 2. Item = (row, 16 codes):
    // consecutive threads read consecutive 16-byte chunks of a row; the 32
    // output bytes are chunks 2c and 2c+1 of the row, XOR-swizzled by row % 8.
    const int ct = tid - 96;
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int r = i % kF8Raw, h = i % kF8Half;
      if (abort_flag || !mbar_wait(&raw_full[r], (i / kF8Raw) & 1) ||
          (i >= kF8Half && !mbar_wait(&half_empty[h], ((i / kF8Half) - 1) & 1))) {
        abort_flag = 1;
        ok = false;
        break;
      }
      const unsigned char* src = sR + r * kF8RawBytes;
      unsigned char* dst = sH + h * kF8HalfBytes;
#pragma unroll
      for (int j = 0; j < kF8Items; ++j) {
        const int item = ct + kF8Conv * j, row = item >> 2, c = item & 3;
        const uint4 w = *reinterpret_cast<const uint4*>(src + row * kTcBK + c * 16);
        uint4 lo, hi;
        lo.x = e4m3x2_to_h2bits(w.x); lo.y = e4m3x2_to_h2bits(w.x >> 16);
        lo.z = e4m3x2_to_h2bits(w.y); lo.w = e4m3x2_to_h2bits(w.y >> 16);
        hi.x = e4m3x2_to_h2bits(w.z); hi.y = e4m3x2_to_h2bits(w.z >> 16);
        hi.z = e4m3x2_to_h2bits(w.w); hi.w = e4m3x2_to_h2bits(w.w >> 16);
        unsigned char* drow = dst + row * 128;
        *reinterpret_cast<uint4*>(drow + (((2 * c) ^ (row & 7)) * 16)) = lo;
        *reinterpret_cast<uint4*>(drow + (((2 * c + 1) ^ (row & 7)) * 16)) = hi;
      }
      fence_async_smem();
      mbar_arrive(&raw_empty[r]);
      mbar_arrive(&half_full[h]);
      if (ct == 0) raw_used_s = i + 1;
    }
    (void)ok;
    pdl_wait();
  }
  __syncwarp();

  // epilogue by warps 3..6 (TMEM lane quarter = warp % 4)
  const bool done_ok = mbar_wait(&done, 0);
  __syncthreads();
  if (tid == 0) have_s = done_ok && !abort_flag && nk > 0;
  __syncthreads();
  tc_fence_after();
  if (warp >= 3 && warp < 7) {
    if (!have_s) {
      if (tid == 96 && (abort_flag || nk > 0)) set_err(a.err, MBT_DEV_WAIT_LIMIT);
    } else {
      tc_epilogue<EPI>(a, tmem, warp & 3, lane, tid - 96, tile, split, sR, 1);   // the raw ring is free now
    }
  }

  // teardown: once `done` fired no MMA is in flight; after a timeout, wait
  // (bounded) for copies that were issued and never consumed
  if (abort_flag && tid == 0) {
    for (int i = raw_used_s; i < raw_issued_s; ++i) mbar_wait(&raw_full[i % kF8Raw], (i / kF8Raw) & 1);
    for (int i = b_used_s; i < b_issued_s; ++i) mbar_wait(&b_full[i % kF8B], (i / kF8B) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tcols) : "memory");
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
