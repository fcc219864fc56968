// Skinny GEMM on the tcgen05 tensor cores for decode at batch 2..64 rows per
// launch, BF16 or e4m3 weights: y = W x with W [rows][K] the M operand
// (swap-AB: 128 weight rows per tile) and the activation rows the N operand.
// BF16 weights: the fp32 activations split into BF16 high and low parts
// (kind::f16). e4m3 weights: the activations split into four e4m3 terms per
// value with a power-of-two scale per row (x = s (c0 + c1/16 + c2/256 +
// c3/4096) to 2^-16 of |x|), multiplied with the weight codes as they are
// (kind::f8f6f4), the 16^-j factors and s applied to the fp32 sums. At these
// batches the weight-only arithmetic intensity 2B / b_w ("GPU Inference
// Internals", "Roofline: Why Decode Is Memory-Bound") is far below the ridge:
// the kernel must move the weights at the HBM rate. Measurements on the GB300
// shape it:
//
// * DRAM efficiency depends on how many contiguous bytes of a weight row one
//   copy fetches: streaming 128-row tiles with TMA boxes of 64 / 128 / 256
//   bytes per row reached 3.9-5.2 / 6.2-6.5 / 6.7 TB/s. Every weight stage
//   here covers 256 bytes of each of its 128 rows (128 BF16 values or 256 e4m3
//   codes), 32 KB per stage.
// * One thread issues a tcgen05.mma about every 100 cycles whatever its N, so
//   the work per instruction decides the MMA rate: at M = 128, N = 128, K = 16
//   (64 cycles of tensor-core time) the issue is the limit. The activation
//   parts are stacked along N (one MMA per K step reads the weight tile once),
//   and e4m3 weights take K = 32 codes per MMA at N = 4 x rows: 8 MMAs per
//   weight stage. The earlier e4m3 design widened the codes to FP16 in TMEM
//   for kind::f16 with FP16 high/low rows, 16 MMAs per stage, and ran at half
//   this kernel's rate.
// * The tensor core's fp32 accumulation drifts toward zero over long chains
//   (a bias proportional to K: 2.3e-5 of the output rms at K = 28672, halving
//   with each halving of the chain). The accumulator therefore lives in TMEM
//   for at most 512 K values: accumulator groups rotate (three for BF16
//   weights, two for e4m3), and the drain warps add the finished one into
//   fp32 registers (IEEE adds) while the MMAs fill the others.
// * Whole tiles per CTA quantise badly (224 tiles on 152 SMs run as two
//   waves). One CTA per SM takes an equal contiguous share of the flattened
//   (tile, K stage) work ("stream-K"). A tile whose K range spans several
//   CTAs belongs to the CTA holding its head (K stage 0): the others did
//   their parts at the start of their shares and published them (coalesced
//   fp32 rows, then a counter), and the owner adds them after its own sums
//   in CTA order, so results do not depend on timing and graph replays match
//   eager runs bit for bit. Under full HBM load one dependent round trip to
//   L2 costs microseconds, so the owner's tail is one acquire and one batch
//   of loads.
//
// Warp roles: warp 0 (one thread) copies weight stages with TMA (it never
// waits on the previous kernel: the weights do not depend on it); warp 1 (one
// thread) copies activation sub-stages (one 128-byte row of K per activation
// row: the high and low rows, or the four term rows); warp 2 (one thread)
// issues the MMAs (columns [x rows, (x + 1) rows) of the accumulator take
// activation part x) and their commits; warp 3 owns the TMEM allocation. The
// last four warps drain the accumulators, finish tiles and run the epilogues:
// split outputs, SwiGLU over 64 gate + 64 up rows (written as 16-bit high/low
// rows for the down projection), the tile's arg-max per row (or the sampling
// draw). Every wait is bounded (about 2 s): on a timeout the kernel flags
// MBT_DEV_WAIT_LIMIT, lets its MMAs and copies finish (bounded), frees TMEM
// and returns.
#include <algorithm>

#include "tcgen05.cuh"

namespace mbt {

constexpr int kTsRows = 64;                        // batch rows per launch (hi + lo = 128 MMA columns)
constexpr int kTsFlushK = 512;                     // K values accumulated in TMEM before the fp32 drain
constexpr uint32_t kTsAStage = 128 * 256;          // weight stage: 128 rows x 256 bytes
constexpr uint32_t kTsRings = 192 * 1024;          // weight ring + activation ring
constexpr uint32_t kTsScratch = 32 * 128 * 4 + 4 * kTsRows * 8;  // epilogue staging (32 batch rows) + arg-max partials
constexpr uint32_t kTsAcc = 64;                    // TMEM columns per accumulator (one per batch row)
constexpr uint32_t kTsTmemCols = 512;

// KSUB: K values per activation sub-stage (one 128-byte row: 64 BF16 values or
// 128 e4m3 codes), SUBS of them per 32 KB weight stage; XR: activation rows per
// batch row (BF16: high and low parts; e4m3: four terms), stacked along N, so
// an accumulator group has XR x 64 TMEM columns; NACC groups rotate; MAXA /
// MAXB: ring depth limits (the depths themselves depend on the batch).
template <int WT> struct TsCfg;
template <> struct TsCfg<W_BF16> {
  static constexpr int KSUB = 64, SUBS = 2, XR = 2, WARPS = 8, DRAIN = 4, MAXA = 5, MAXB = 8, NACC = 3;
};
template <> struct TsCfg<W_E4M3> {
  static constexpr int KSUB = 128, SUBS = 2, XR = 4, WARPS = 8, DRAIN = 4, MAXA = 4, MAXB = 16, NACC = 2;
};

constexpr size_t ts_smem() { return 1024 + (size_t)kTsRings + kTsScratch; }

// Ring depths for Rc padded batch rows. Under full HBM load an activation
// copy from L2 takes as long as a weight copy from HBM (3,400-7,000 cycles
// measured against 6,000), so both rings are sized against that latency: the
// activation bytes per weight byte are 4 Rc / (128 w) (four bytes per value:
// two BF16 parts or four e4m3 terms), and the rings split the 192 KB in
// roughly that proportion.
template <int WT>
__host__ __device__ __forceinline__ void ts_rings(int Rc, int& sa, int& sb) {
  using C = TsCfg<WT>;
  const int xs = C::XR * Rc * 128;
  sa = WT == W_E4M3 ? (Rc <= 16 ? 4 : 3) : (Rc <= 16 ? 5 : 4);
  if (sa > C::MAXA) sa = C::MAXA;
  sb = ((int)kTsRings - sa * (int)kTsAStage) / xs;
  if (sb > C::MAXB) sb = C::MAXB;
}

// First unit (weight stage) of CTA c's share of W units over G CTAs.
__device__ __forceinline__ long long ts_u0(long long W, int G, int c) { return W * c / G; }
// The CTA whose share holds unit u.
__device__ __forceinline__ int ts_owner(long long W, int G, long long u) {
  int c = (int)((u * G) / W);
  while (c + 1 < G && ts_u0(W, G, c + 1) <= u) ++c;
  while (c > 0 && ts_u0(W, G, c) > u) --c;
  return c;
}

// silu(x) = x / (1 + e^-x) with the hardware exponential and divide
// (a few ulp; exact limits: 0 for x -> -inf, x for x -> +inf).
__device__ __forceinline__ float ts_silu(float x) { return __fdividef(x, 1.f + __expf(-x)); }

// x = hi + lo as 16-bit bit patterns (FP16 or BF16), the same rounding as store_hl16.
__device__ __forceinline__ void split_hl16(float x, int f16, uint32_t& hi, uint32_t& lo) {
  if (f16) {
    const __half h = __float2half_rn(x);
    hi = __half_as_ushort(h);
    lo = __half_as_ushort(__float2half_rn(x - __half2float(h)));
  } else {
    const bf16 h = __float2bfloat16_rn(x);
    hi = __bfloat16_as_ushort(h);
    lo = __bfloat16_as_ushort(__float2bfloat16_rn(x - __bfloat162float(h)));
  }
}

template <int WT, int EPI>
__global__ void __launch_bounds__(TsCfg<WT>::WARPS * 32, 1)
tc_stream_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const TcArgs a) {
  using C = TsCfg<WT>;
  constexpr int SUBS = C::SUBS, KSUB = C::KSUB, XR = C::XR;
  constexpr int ACOLS = XR * kTsAcc;                 // TMEM columns per accumulator group
  constexpr int FG = kTsFlushK / (KSUB * SUBS);      // weight stages per accumulation group
  constexpr int DW = C::DRAIN;                       // first drain warp
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t a_full[C::MAXA], a_empty[C::MAXA], b_full[C::MAXB], b_empty[C::MAXB];
  __shared__ __align__(8) uint64_t acc_full[C::NACC], acc_empty[C::NACC], done;
  __shared__ float xsc_s[kTsRows];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ int a_issued_s, a_used_s, b_issued_s, b_used_s, last_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int Rc = a.Rp;                                // padded rows of this launch (multiple of 16, <= 64)
  int SA, SB;
  ts_rings<WT>(Rc, SA, SB);
  const uint32_t b_bytes = (uint32_t)(XR * Rc) * 128;       // one activation sub-stage
  unsigned char* sA = smem;                                   // [SA][K block][128 rows][128 B], 128-B swizzle
  unsigned char* sB = sA + SA * kTsAStage;                    // [SB][XR * Rc rows][128 B], 128-B swizzle
  float* scr = reinterpret_cast<float*>(smem + kTsRings);     // epilogue staging
  const int tiles = EPI == EPI_SWIGLU ? (a.N + 63) / 64 : (a.N + 127) / 128;
  const int nA = (a.K + KSUB * SUBS - 1) / (KSUB * SUBS);
  const long long W = (long long)tiles * nA;
  const long long u0 = ts_u0(W, G, cta), u1 = ts_u0(W, G, cta + 1);
  auto rowA0 = [&](int t) { return EPI == EPI_SWIGLU ? t * 64 : t * 128; };
  auto rowA1 = [&](int t) { return EPI == EPI_SWIGLU ? a.N + t * 64 : t * 128 + 64; };

  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < SA; ++s) { mbar_init(&a_full[s], 1); mbar_init(&a_empty[s], 1); }
    for (int s = 0; s < SB; ++s) { mbar_init(&b_full[s], 1); mbar_init(&b_empty[s], 1); }
    for (int s = 0; s < C::NACC; ++s) { mbar_init(&acc_full[s], 1); mbar_init(&acc_empty[s], 4); }
    mbar_init(&done, 1);
    abort_flag = 0;
    a_issued_s = a_used_s = b_issued_s = b_used_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
  }
  if (warp == 3) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(&tmem_slot)), "r"(kTsTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;                      // accumulator groups at columns 0, ACOLS, ...

  if (warp == 0) {
    if (lane == 0) {
      // weight stages of this CTA's units, in order
      int i = 0, s = 0, r = 0;                         // copy count, its slot and round
      for (long long u = u0; u < u1; ++u, ++i, s = s + 1 == SA ? 0 : s + 1, r += s == 0) {
        if (r > 0 && (abort_flag || !mbar_wait(&a_empty[s], (uint32_t)((r - 1) & 1)))) { abort_flag = 1; break; }
        const int t = (int)(u / nA), k = (int)(u % nA);
        mbar_arrive_tx(&a_full[s], kTsAStage);
        unsigned char* dst = sA + (size_t)s * kTsAStage;
#pragma unroll
        for (int h = 0; h < 2; ++h) {                 // two 128-byte K blocks of each row
          const int kx = WT == W_E4M3 ? k * 256 + h * 128 : (k * 2 + h) * 64;
          tma_load_2d(dst + h * 16384, &tmW, kx, rowA0(t), &a_full[s]);
          tma_load_2d(dst + h * 16384 + 8192, &tmW, kx, rowA1(t), &a_full[s]);
        }
        a_issued_s = i + 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      pdl_wait();
      int i = 0, s = 0, r = 0;
      for (long long u = u0; u < u1 && !abort_flag; ++u) {
        const int k = (int)(u % nA);
        for (int j = 0; j < SUBS; ++j, ++i, s = s + 1 == SB ? 0 : s + 1, r += s == 0) {
          if (r > 0 && (abort_flag || !mbar_wait(&b_empty[s], (uint32_t)((r - 1) & 1)))) { abort_flag = 1; break; }
          const int kx = (k * SUBS + j) * KSUB;
          mbar_arrive_tx(&b_full[s], b_bytes);
          unsigned char* dst = sB + (size_t)s * b_bytes;
#pragma unroll
          for (int x = 0; x < XR; ++x)                 // high / low rows, or the four term rows
            tma_load_2d(dst + (size_t)x * Rc * 128, &tmX, kx, x * a.rp_all + a.row0, &b_full[s]);
          b_issued_s = i + 1;
        }
      }
    }
  } else if (warp == 2) {
    if (lane == 0) {
      pdl_wait();
      // M = 128 weight rows, N = XR x Rc activation rows (K = 16 BF16 values or
      // 32 e4m3 codes per MMA, four MMAs per sub-stage)
      const uint32_t idesc = idesc_16(128, XR * Rc, WT == W_E4M3 ? 1 : 0);
      int ia = 0, sa = 0, ra = 0, ib = 0, sb = 0, rb = 0, gi = 0;   // counts, slots, rounds
      bool ok = true;
      for (long long u = u0; u < u1 && ok;) {
        const int k0 = (int)(u % nA);
        const int seg = (int)min((long long)(nA - k0), u1 - u);
        for (int g0 = 0; g0 < seg && ok; g0 += FG, ++gi) {
          const int gn = min(FG, seg - g0);
          const int buf = gi % C::NACC;
          if (gi >= C::NACC && !mbar_wait(&acc_empty[buf], (uint32_t)(((gi / C::NACC) - 1) & 1))) { ok = false; break; }
          tc_fence_after();
          const uint32_t acc = tmem + (uint32_t)(buf * ACOLS);   // columns [x Rc, (x + 1) Rc): activation part x
          for (int x = 0; x < gn && ok; ++x, ++ia, sa = sa + 1 == SA ? 0 : sa + 1, ra += sa == 0) {
            if (abort_flag || !mbar_wait(&a_full[sa], (uint32_t)(ra & 1))) { ok = false; break; }
            for (int j = 0; j < SUBS; ++j, ++ib, sb = sb + 1 == SB ? 0 : sb + 1, rb += sb == 0) {
              if (abort_flag || !mbar_wait(&b_full[sb], (uint32_t)(rb & 1))) { ok = false; break; }
              tc_fence_after();
              const uint64_t bh = sw128_desc(smem_u32(sB + (size_t)sb * b_bytes));
              const uint64_t ad = sw128_desc(smem_u32(sA + (size_t)sa * kTsAStage + j * 16384));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {             // 32 bytes of K per MMA
                const uint32_t accum = (x > 0 || j > 0 || kk > 0) ? 1u : 0u;
                if (WT == W_E4M3) umma_kf8(acc, ad + (uint64_t)(kk * 2), bh + (uint64_t)(kk * 2), idesc, accum);
                else umma_kf16(acc, ad + (uint64_t)(kk * 2), bh + (uint64_t)(kk * 2), idesc, accum);
              }
              umma_commit(&b_empty[sb]);
              b_used_s = ib + 1;
            }
            if (ok) { umma_commit(&a_empty[sa]); a_used_s = ia + 1; }
          }
          if (ok) umma_commit(&acc_full[buf]);
        }
        u += seg;
      }
      if (!ok) abort_flag = 1;
      umma_commit(&done);                              // fires once every MMA issued above has completed
    }
  } else if (warp >= DW) {
    // drain, finish and epilogue: thread = weight row q * 32 + lane of the tile.
    // The tile counters and partial sums are shared with the previous launch
    // on the stream: nothing here touches them before that launch is done.
    pdl_wait();
    const int q = warp - DW, row = q * 32 + lane, et = tid - DW * 32;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    if (WT == W_E4M3) {                                // the term rows' scales, for the epilogue
      if (et < kTsRows) xsc_s[et] = et < Rc ? a.x_scale[a.row0 + et] : 1.f;
      named_bar(3, 128);
    }
    float sum[kTsRows];
    int gi = 0;
    bool ok = true;
    for (long long u = u0; u < u1 && ok;) {
      const int t = (int)(u / nA), k0 = (int)(u % nA);
      const int seg = (int)min((long long)(nA - k0), u1 - u);
#pragma unroll
      for (int b = 0; b < kTsRows; ++b) sum[b] = 0.f;
      // the head of a cut tile: read the tile's counter while the last MMAs
      // still run (the other contributors published long ago, as a rule)
      const bool owned = k0 == 0 && seg < nA;
      int early = -1;
      for (int g0 = 0; g0 < seg; g0 += FG, ++gi) {
        const int buf = gi % C::NACC;
        if (owned && et == 0 && g0 + FG >= seg) early = ld_acquire_gpu(a.ts_tickets + t);
        if (abort_flag || !mbar_wait(&acc_full[buf], (uint32_t)((gi / C::NACC) & 1))) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int part = 0; part < XR; ++part) {          // high then low rows, or term 0..3
          // term x carries 16^-x of the row's scale (exact power-of-two factors)
          const float f = WT == W_E4M3 ? (part == 0 ? 1.f : part == 1 ? 0.0625f : part == 2 ? 0.00390625f : 0.000244140625f) : 1.f;
          const uint32_t acc = tmem + (uint32_t)(buf * ACOLS) + (uint32_t)(part * Rc) + lane_base;
          // all of the row's columns in flight at once, one wait
          uint32_t v0[16], v1[16], v2[16], v3[16];
          tmem_ld16_async(acc, v0);
          if (Rc > 16) tmem_ld16_async(acc + 16, v1);
          if (Rc > 32) tmem_ld16_async(acc + 32, v2);
          if (Rc > 48) tmem_ld16_async(acc + 48, v3);
          tmem_ld_wait16(v0);
          tmem_ld_wait16(v1);
          tmem_ld_wait16(v2);
          tmem_ld_wait16(v3);
          if (WT == W_E4M3) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              sum[j] += __uint_as_float(v0[j]) * f;
              if (Rc > 16) sum[16 + j] += __uint_as_float(v1[j]) * f;
              if (Rc > 32) sum[32 + j] += __uint_as_float(v2[j]) * f;
              if (Rc > 48) sum[48 + j] += __uint_as_float(v3[j]) * f;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              sum[j] += __uint_as_float(v0[j]);
              if (Rc > 16) sum[16 + j] += __uint_as_float(v1[j]);
              if (Rc > 32) sum[32 + j] += __uint_as_float(v2[j]);
              if (Rc > 48) sum[48 + j] += __uint_as_float(v3[j]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      }
      if (!ok) break;
      const bool whole = k0 == 0 && seg == nA;
      if (!whole) {
        // A tile cut by a share boundary. A share can only begin inside a
        // tile, so the part of a tile that is not its head is always the
        // first segment of its CTA, done early: those CTAs publish their sums
        // and move on. The CTA holding the head of the tile (its last segment,
        // or a head that ends its share) owns the tile: it waits for the
        // others (bounded), adds their sums after its own in CTA order (the
        // same order on every run) and runs the epilogue.
        const int c_first = ts_owner(W, G, (long long)t * nA);
        const int c_last = ts_owner(W, G, (long long)t * nA + nA - 1);
        if (k0 != 0) {
          float* mine = a.ts_scratch + (size_t)cta * 128 * kTsRows + row;   // [row b][weight row]
#pragma unroll
          for (int b = 0; b < kTsRows; ++b) if (b < Rc) mine[(size_t)b * 128] = sum[b];
          __threadfence();
          named_bar(1, 128);
          if (et == 0) atomicAdd(a.ts_tickets + t, 1);
          u += seg;
          continue;
        }
        if (et == 0) {
          const int want = c_last - c_first;
          int seen = early >= want ? early : ld_acquire_gpu(a.ts_tickets + t);
          if (seen < want) {
            const long long w0 = clock64();
            while ((seen = ld_acquire_gpu(a.ts_tickets + t)) < want && clock64() - w0 < kTcWaitCycles) {}
          }
          last_s = seen == want;
        }
        named_bar(1, 128);
        if (!last_s) { ok = false; break; }
        for (int cc = c_first + 1; cc <= c_last; ++cc) {
          const float* src = a.ts_scratch + (size_t)cc * 128 * kTsRows + row;
          float p[kTsRows];
#pragma unroll
          for (int b = 0; b < kTsRows; ++b) p[b] = b < Rc ? __ldcg(src + (size_t)b * 128) : 0.f;
#pragma unroll
          for (int b = 0; b < kTsRows; ++b) sum[b] += p[b];
        }
        if (et == 0) a.ts_tickets[t] = 0;              // every contributor has arrived: ready for the next launch
      }
      // ---- epilogue of tile t. The scaled sums pass through shared memory
      // ([batch row][weight row], conflict-free) in two halves of 32 batch
      // rows and are consumed by rolled loops: epilogues unrolled over the 64
      // rows were tens of KB of instructions, fetched cold once per tile, and
      // under full HBM load that cost ~300 cycles per batch row at the tail.
      float sc;
      if (EPI == EPI_SWIGLU) {
        const int j = t * 64 + (row & 63);              // rows 0..63: gate, 64..127: up of channel j
        sc = (a.scale && j < a.N) ? a.scale[row < 64 ? j : a.N + j] : 1.f;
      } else {
        const int n = t * 128 + row;
        sc = (a.scale && n < a.N) ? a.scale[n] : 1.f;
      }
      float* bv = scr + 32 * 128;                        // arg-max: [4 warps][kTsRows] best value, index
      int* bi = reinterpret_cast<int*>(bv + 4 * kTsRows);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b0 = h * 32;
        if (b0 >= Rc) break;
        named_bar(2, 128);                               // the staging buffer is free
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (b0 + i < Rc) scr[i * 128 + row] = sum[b0 + i] * (WT == W_E4M3 ? sc * xsc_s[b0 + i] : sc);
        named_bar(2, 128);
        const int nb = min(32, Rc - b0);
        if (EPI == EPI_PARTIAL) {
          // four consecutive outputs of one batch row per thread and pass
          const bool vec = ((a.ldo & 3) == 0) && (((uintptr_t)a.out & 15) == 0);
          for (int e = et; e < nb * 32; e += 128) {
            const int i = e >> 5, n4 = (e & 31) * 4, b = b0 + i, n = t * 128 + n4;
            if (b >= a.R || n >= a.N) continue;
            const float4 v = *reinterpret_cast<const float4*>(scr + i * 128 + n4);
            float* o = a.out + (size_t)(a.row0 + b) * a.ldo + n;
            if (vec && n + 3 < a.N) {
              *reinterpret_cast<float4*>(o) = v;
            } else {
              o[0] = v.x;
              if (n + 1 < a.N) o[1] = v.y;
              if (n + 2 < a.N) o[2] = v.z;
              if (n + 3 < a.N) o[3] = v.w;
            }
          }
        } else if (EPI == EPI_SWIGLU) {
          // four consecutive channels of one batch row per thread and pass,
          // written as 8-byte high and low words
          uint16_t* act = reinterpret_cast<uint16_t*>(a.act_hl);
          const bool vec = (a.ld_act & 3) == 0;
          for (int e = et; e < nb * 16; e += 128) {
            const int i = e >> 4, c4 = (e & 15) * 4, j = t * 64 + c4, b = b0 + i;
            if (j >= a.N) continue;
            const float4 g = *reinterpret_cast<const float4*>(scr + i * 128 + c4);
            const float4 u = *reinterpret_cast<const float4*>(scr + i * 128 + 64 + c4);
            const bool live = b < a.R;                    // padding rows stay finite (zero)
            const float v[4] = {live ? ts_silu(g.x) * u.x : 0.f, live ? ts_silu(g.y) * u.y : 0.f,
                                live ? ts_silu(g.z) * u.z : 0.f, live ? ts_silu(g.w) * u.w : 0.f};
            uint16_t* hi = act + (size_t)(a.row0 + b) * a.ld_act + j;
            uint16_t* lo = act + (size_t)(a.rp_all + a.row0 + b) * a.ld_act + j;
            if (vec && j + 3 < a.N) {
              uint32_t h[4], l[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) split_hl16(v[q], a.hl_f16, h[q], l[q]);
              *reinterpret_cast<uint2*>(hi) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
              *reinterpret_cast<uint2*>(lo) = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
            } else {
              for (int q = 0; q < 4 && j + q < a.N; ++q) store_hl16(hi + q, lo + q, v[q], a.hl_f16);
            }
          }
        } else {  // EPI_ARGMAX: the tile's best (value, index) per batch row
          const int n = t * 128 + row;
          for (int i = 0; i < nb; ++i) {
            const int b = b0 + i;
            float v = n < a.N ? scr[i * 128 + row] : -INFINITY;
            if (!(v == v)) { set_err(a.err, MBT_DEV_NONFINITE); v = -INFINITY; }
            if (n < a.N && b < a.R && a.logits) a.logits[(size_t)(a.row0 + b) * a.ldl + n] = v;
            if (a.gum.on && n < a.N) v = gumbel_score(v, n, b, a.gum);
            int idx = n;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              const float ov = __shfl_xor_sync(0xffffffffu, v, o);
              const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
              if (ov > v || (ov == v && oi < idx)) { v = ov; idx = oi; }
            }
            if (lane == 0) { bv[q * kTsRows + b] = v; bi[q * kTsRows + b] = idx; }
          }
        }
      }
      if (EPI == EPI_ARGMAX) {
        named_bar(2, 128);
        for (int b = et; b < a.R; b += 128) {
          float v = bv[b];
          int idx = bi[b];
          for (int w2 = 1; w2 < 4; ++w2) {
            const float ov = bv[w2 * kTsRows + b];
            const int oi = bi[w2 * kTsRows + b];
            if (ov > v || (ov == v && oi < idx)) { v = ov; idx = oi; }
          }
          ArgmaxPart p;
          p.v = v; p.i = idx;
          a.part[(size_t)t * a.part_ld + a.row0 + b] = p;
        }
      }
      u += seg;
    }
    if (!ok) abort_flag = 1;
  }
  __syncwarp();

  // teardown: `done` covers every MMA; after a timeout, wait (bounded) for the
  // copies that were issued and never consumed before shared memory goes
  const bool done_ok = mbar_wait(&done, 0);
  __syncthreads();
  if (tid == 0 && (abort_flag || !done_ok)) {
    set_err(a.err, MBT_DEV_WAIT_LIMIT);
    for (int i = a_used_s; i < a_issued_s; ++i) mbar_wait(&a_full[i % SA], (uint32_t)((i / SA) & 1));
    for (int i = b_used_s; i < b_issued_s; ++i) mbar_wait(&b_full[i % SB], (uint32_t)((i / SB) & 1));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 3) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTsTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// host side

namespace {
template <int WT, int EPI>
void* ts_fn() { return (void*)tc_stream_kernel<WT, EPI>; }
template <int WT>
void* ts_pick_w(int epi) {
  return epi == EPI_PARTIAL ? ts_fn<WT, EPI_PARTIAL>() : epi == EPI_SWIGLU ? ts_fn<WT, EPI_SWIGLU>()
                                                                            : ts_fn<WT, EPI_ARGMAX>();
}
void* ts_pick(int wt, int epi) { return wt == W_E4M3 ? ts_pick_w<W_E4M3>(epi) : ts_pick_w<W_BF16>(epi); }
}  // namespace

cudaError_t ts_init() {
  for (int wt = 0; wt < 2; ++wt)
    for (int epi = 0; epi < 3; ++epi) {
      const size_t sm = ts_smem();
      cudaError_t e = cudaFuncSetAttribute(ts_pick(wt, epi), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

int ts_tiles(int epi, int N) { return epi == EPI_SWIGLU ? (N + 63) / 64 : (N + 127) / 128; }

size_t ts_scratch_floats(int num_sms) { return (size_t)num_sms * 128 * kTsRows; }

cudaError_t ts_launch(int wt, int epi, const void* mapW, const void* mapX, const TcArgs& a, int num_sms,
                      cudaStream_t s) {
  if (a.Rp < 16 || a.Rp > kTsRows || a.Rp % 16 || a.R < 1 || a.R > a.Rp || a.rp_all < a.row0 + a.Rp ||
      !a.ts_scratch || !a.ts_tickets || a.tickets_cap < ts_tiles(epi, a.N) || (wt == W_E4M3 && !a.x_scale))
    return cudaErrorInvalidValue;
  CUtensorMap w = *(const CUtensorMap*)mapW, x = *(const CUtensorMap*)mapX;
  TcArgs args = a;
  args.gum.row0 += a.row0;
  void* params[] = {&w, &x, &args};
  const int threads = (wt == W_E4M3 ? TsCfg<W_E4M3>::WARPS : TsCfg<W_BF16>::WARPS) * 32;
  const size_t sm = ts_smem();
  // one CTA per SM, but never more CTAs than weight stages: every CTA's share
  // is then non-empty, so a tile's contributors are consecutive CTAs
  const int kst = wt == W_E4M3 ? TsCfg<W_E4M3>::SUBS * TsCfg<W_E4M3>::KSUB : TsCfg<W_BF16>::SUBS * TsCfg<W_BF16>::KSUB;
  const long long units = (long long)ts_tiles(epi, a.N) * ((a.K + kst - 1) / kst);
  const int grid = (int)std::min<long long>(num_sms, units);
  return launch_pdl(ts_pick(wt, epi), dim3(grid), dim3(threads), sm, s, params);
}

}  // namespace mbt
