// Weight-streaming GEMV for decode at batch 1..8 (CUDA cores).
//
// Decode "is effectively a matrix-vector product: it reads enormous weight
// matrices to compute a single token's worth of output" ("Kernel Fusion for
// Large-Scale LLM Inference", section 10), so the kernel is built around one
// pass over the weights at the HBM rate:
//   * every weight byte is loaded once with 16-byte streaming loads (L1 bypass),
//     a warp instruction covering 512 contiguous bytes of one row, several rows
//     and vectors per thread in flight;
//   * the activation rows x (BF16) sit in shared memory for the whole CTA;
//   * rows are split over CTAs in equal contiguous ranges (the grid is a
//     multiple of the SM count), so every SM streams the same number of bytes;
//   * FP8-e4m3 weights are converted in registers and the per-output-channel
//     scale is applied once to the finished dot product, which is exact
//     reassociation ("Epilogue and dequant fusion", same section 11);
//   * three epilogues: fp32 partial sums (split-K), the SwiGLU activation over
//     the fused gate/up rows ("Kernels, Fusion & CUDA Graphs", "Fix 1: kernel
//     fusion": gate + up projection and SiLU x mul), and a per-CTA arg-max over
//     LM-head rows so that logits need not reach HBM (same table, "Sampling").
#include "common.cuh"
#include "internal.h"

namespace mbt {

template <int NB> struct GemvShape;
template <> struct GemvShape<1> { static constexpr int RG = 8, U = 2, MINB = 2; };
template <> struct GemvShape<2> { static constexpr int RG = 8, U = 2, MINB = 2; };
template <> struct GemvShape<4> { static constexpr int RG = 4, U = 2, MINB = 2; };
template <> struct GemvShape<8> { static constexpr int RG = 4, U = 2, MINB = 1; };

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;

// Reduce M per-lane values over the warp with a transpose: each step halves the
// values a lane keeps, so M values cost about M shuffles instead of 5 M. On
// return the lane holds the warp total of value `idx`.
template <int M>
__device__ __forceinline__ float warp_transpose_sum(float (&v)[M], int lane, int& idx) {
  idx = 0;
  int m = M;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (m > 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int j = 0; j < M / 2; ++j) {
        if (j < m / 2) {
          const float send = upper ? v[j] : v[j + m / 2];
          const float keep = upper ? v[j + m / 2] : v[j];
          v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      if (upper) idx += m / 2;
      m >>= 1;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  return v[0];
}

template <int WT>
__device__ __forceinline__ void widen8(const uint4& w, int half, float (&f)[8]);

template <>
__device__ __forceinline__ void widen8<W_BF16>(const uint4& w, int, float (&f)[8]) {
  f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
  f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

template <>
__device__ __forceinline__ void widen8<W_E4M3>(const uint4& w, int half, float (&f)[8]) {
  const uint32_t a = half ? w.z : w.x, b = half ? w.w : w.y;
  float2 t;
  t = e4m3x2_to_float2(a);        f[0] = t.x; f[1] = t.y;
  t = e4m3x2_to_float2(a >> 16);  f[2] = t.x; f[3] = t.y;
  t = e4m3x2_to_float2(b);        f[4] = t.x; f[5] = t.y;
  t = e4m3x2_to_float2(b >> 16);  f[6] = t.x; f[7] = t.y;
}

template <int NB, int WT, int EPI>
__global__ void __launch_bounds__(kGemvThreads, GemvShape<NB>::MINB)
gemv_kernel(const GemvArgs a) {
  constexpr int RG = GemvShape<NB>::RG;          // weight rows per group
  constexpr int U = GemvShape<NB>::U;            // 16-B vectors per row per thread in flight
  constexpr int EPV = (WT == W_BF16) ? 8 : 16;   // elements per 16-B weight vector
  constexpr int HALVES = EPV / 8;                // 8-element halves per vector
  constexpr int M = RG * NB;                     // dot products per group
  constexpr int CH = (EPI == EPI_SWIGLU) ? RG / 2 : RG;   // output channels per group
  static_assert(M <= 32 && (M & (M - 1)) == 0, "M must be a power of two <= 32");

  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // this CTA's split of K, in 16-byte weight vectors
  const int nvec_all = a.K / EPV;
  const int split = blockIdx.y, nsplit = gridDim.y;
  const int v0 = (int)((long long)nvec_all * split / nsplit);
  const int nvec = (int)((long long)nvec_all * (split + 1) / nsplit) - v0;

  // x tile: [NB][HALVES][nvec] uint4 (8 BF16 each): thread-contiguous reads
  uint4* xs = reinterpret_cast<uint4*>(smem);
  const int xrow = nvec * HALVES;
  float* red = reinterpret_cast<float*>(smem + (size_t)NB * xrow * 16);   // [2][warps][32]
  float* fin = red + 2 * kGemvWarps * 32;                                  // [M]
  {
    const bf16* xb = a.x + (size_t)v0 * EPV;
    for (int i = tid; i < NB * xrow; i += kGemvThreads) {
      const int b = i / xrow, j = i - b * xrow;          // j = h * nvec + v
      const int h = j / nvec, v = j - h * nvec;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (b < a.nb) val = *reinterpret_cast<const uint4*>(xb + (size_t)b * a.ldx + (size_t)v * EPV + h * 8);
      xs[i] = val;
    }
  }
  __syncthreads();

  const int G = gridDim.x, c = blockIdx.x;
  const int r_begin = (int)((long long)a.N * c / G);
  const int r_end = (int)((long long)a.N * (c + 1) / G);
  const size_t row_bytes = (size_t)a.K * (WT == W_BF16 ? 2 : 1);
  const unsigned char* Wb = reinterpret_cast<const unsigned char*>(a.W) + (size_t)v0 * 16;

  float best_v = -INFINITY;
  int best_i = 0x7fffffff;
  int buf = 0;

  for (int r0 = r_begin; r0 < r_end; r0 += CH, buf ^= 1) {
    const unsigned char* rowp[RG];
#pragma unroll
    for (int i = 0; i < RG; ++i) {
      int ch = r0 + (i % CH);
      ch = ch < r_end ? ch : r_end - 1;
      const int wr = (EPI == EPI_SWIGLU && i >= CH) ? a.N + ch : ch;
      rowp[i] = Wb + (size_t)wr * row_bytes;
    }
    float acc[M];
#pragma unroll
    for (int j = 0; j < M; ++j) acc[j] = 0.f;

    for (int v = tid; v < nvec; v += kGemvThreads * U) {
      uint4 w[U][RG];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int vv = v + u * kGemvThreads;
#pragma unroll
        for (int i = 0; i < RG; ++i)
          w[u][i] = vv < nvec ? ld_stream(rowp[i] + (size_t)vv * 16) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int vv = v + u * kGemvThreads;
        if (vv < nvec) {
#pragma unroll
          for (int h = 0; h < HALVES; ++h) {
            float xf[NB][8];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              const uint4 xv = xs[b * xrow + h * nvec + vv];
              widen8<W_BF16>(xv, 0, xf[b]);
            }
#pragma unroll
            for (int i = 0; i < RG; ++i) {
              float wf[8];
              widen8<WT>(w[u][i], h, wf);
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                float s = acc[i * NB + b];
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(wf[e], xf[b][e], s);
                acc[i * NB + b] = s;
              }
            }
          }
        }
      }
    }

    // CTA reduction of the M dot products
    int idx;
    const float part = warp_transpose_sum<M>(acc, lane, idx);
    float* rb = red + buf * kGemvWarps * 32;
    if ((lane & (32 / M - 1)) == 0) rb[warp * 32 + idx] = part;
    __syncthreads();

    if (EPI == EPI_PARTIAL) {
      if (tid < M) {
        const int i = tid / NB, b = tid % NB, ch = r0 + i;
        float t = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kGemvWarps; ++w2) t += rb[w2 * 32 + tid];
        if (ch < r_end && b < a.nb) {
          if (WT == W_E4M3) t *= a.scale[ch];
          a.out[(size_t)split * a.split_stride + (size_t)b * a.ldo + ch] = t;
        }
      }
    } else if (EPI == EPI_SWIGLU) {
      if (tid < CH * NB) {
        const int i = tid / NB, b = tid % NB, ch = r0 + i;
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kGemvWarps; ++w2) {
          g += rb[w2 * 32 + tid];
          u += rb[w2 * 32 + tid + CH * NB];
        }
        if (ch < r_end && b < a.nb) {
          if (WT == W_E4M3) { g *= a.scale[ch]; u *= a.scale[a.N + ch]; }
          const float act = g / (1.f + expf(-g)) * u;
          a.act[(size_t)b * a.lda + ch] = __float2bfloat16_rn(act);
        }
      }
    } else {  // EPI_ARGMAX
      if (tid < M) {
        const int i = tid / NB, b = tid % NB, ch = r0 + i;
        float t = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kGemvWarps; ++w2) t += rb[w2 * 32 + tid];
        if (WT == W_E4M3 && ch < r_end) t *= a.scale[ch];
        fin[tid] = t;
        if (ch < r_end && b < a.nb && a.logits) a.logits[(size_t)b * a.ldl + ch] = t;
      }
      __syncthreads();
      if (tid < NB) {
#pragma unroll
        for (int i = 0; i < RG; ++i) {
          const int ch = r0 + i;
          if (ch < r_end) {
            const float t = fin[i * NB + tid];
            if (t > best_v) { best_v = t; best_i = ch; }          // rows ascend: first max kept
            else if (!(t == t)) set_err(a.err, MBT_DEV_NONFINITE);
          }
        }
      }
    }
  }
  if (EPI == EPI_ARGMAX && tid < NB && tid < a.nb) {
    ArgmaxPart p; p.v = best_v; p.i = best_i;
    a.part[(size_t)c * a.part_ld + tid] = p;
  }
}

// ---------------------------------------------------------------------------
// host side

namespace {
constexpr size_t kXsBudgetShared = 96 * 1024;    // 2 CTAs per SM
constexpr size_t kXsBudgetSolo = 192 * 1024;     // 1 CTA per SM (NB = 8)

int nb_template(int nb) { return nb <= 1 ? 1 : nb <= 2 ? 2 : nb <= 4 ? 4 : 8; }

template <int NB>
int group_rows(int epi) { return epi == EPI_SWIGLU ? GemvShape<NB>::RG / 2 : GemvShape<NB>::RG; }

int rows_per_group(int nbt, int epi) {
  switch (nbt) {
    case 1: return group_rows<1>(epi);
    case 2: return group_rows<2>(epi);
    case 4: return group_rows<4>(epi);
    default: return group_rows<8>(epi);
  }
}

template <int NB, int WT, int EPI>
void* kernel_ptr() { return (void*)gemv_kernel<NB, WT, EPI>; }

void* pick(int nbt, int wt, int epi) {
#define MBT_PICK_E(NB, WT)                                               \
  switch (epi) {                                                         \
    case EPI_PARTIAL: return kernel_ptr<NB, WT, EPI_PARTIAL>();          \
    case EPI_SWIGLU: return kernel_ptr<NB, WT, EPI_SWIGLU>();            \
    default: return kernel_ptr<NB, WT, EPI_ARGMAX>();                    \
  }
#define MBT_PICK_W(NB) \
  if (wt == W_BF16) { MBT_PICK_E(NB, W_BF16) } else { MBT_PICK_E(NB, W_E4M3) }
  switch (nbt) {
    case 1: MBT_PICK_W(1)
    case 2: MBT_PICK_W(2)
    case 4: MBT_PICK_W(4)
    default: MBT_PICK_W(8)
  }
#undef MBT_PICK_W
#undef MBT_PICK_E
}
}  // namespace

GemvLaunch gemv_plan(int epi, int wtype, int nb, int N, int K, int num_sms, int force_nsplit) {
  GemvLaunch g;
  g.nb_tmpl = nb_template(nb);
  const int epv = wtype == W_BF16 ? 8 : 16;
  const int nvec_all = K / epv;
  const size_t budget = g.nb_tmpl == 8 ? kXsBudgetSolo : kXsBudgetShared;
  const size_t xs_full = (size_t)g.nb_tmpl * K * 2;
  int ns = (int)((xs_full + budget - 1) / budget);
  if (epi != EPI_PARTIAL) ns = 1;
  if (force_nsplit > 0) ns = force_nsplit;
  if (ns > nvec_all) ns = nvec_all;
  if (ns < 1) ns = 1;
  g.nsplit = ns;
  const int per_sm = g.nb_tmpl == 8 ? 1 : 2;
  int grid = num_sms * per_sm / ns;
  if (grid < 1) grid = 1;
  const int rg = rows_per_group(g.nb_tmpl, epi);
  const int max_grid = (N + rg - 1) / rg;
  if (grid > max_grid) grid = max_grid;
  g.grid = grid;
  const size_t nvec_max = (size_t)(nvec_all + ns - 1) / ns;
  g.smem = (size_t)g.nb_tmpl * nvec_max * 16 * (epv / 8) + 2 * kGemvWarps * 32 * 4 + 32 * 4;
  return g;
}

cudaError_t gemv_launch(int epi, const GemvArgs& a, const GemvLaunch& g, cudaStream_t s) {
  void* fn = pick(g.nb_tmpl, a.wtype, epi);
  GemvArgs args = a;
  void* params[] = {&args};
  return cudaLaunchKernel(fn, dim3(g.grid, g.nsplit), dim3(kGemvThreads), params, g.smem, s);
}

cudaError_t gemv_init() {
  const int nbs[4] = {1, 2, 4, 8};
  for (int i = 0; i < 4; ++i)
    for (int wt = 0; wt < 2; ++wt)
      for (int epi = 0; epi < 3; ++epi) {
        const int lim = nbs[i] == 8 ? 227 * 1024 : 113 * 1024;
        cudaError_t e = cudaFuncSetAttribute(pick(nbs[i], wt, epi),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
        if (e != cudaSuccess) return e;
      }
  return cudaSuccess;
}

}  // namespace mbt
