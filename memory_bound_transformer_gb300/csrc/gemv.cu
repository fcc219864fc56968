// Weight-streaming GEMV for decode at batch 1..15 (CUDA cores; up to 8 rows per launch).
//
// Decode "is effectively a matrix-vector product: it reads enormous weight
// matrices to compute a single token's worth of output" ("Kernel Fusion for
// Large-Scale LLM Inference", section 10), so the kernel is built around one
// pass over the weights at the HBM rate:
//   * every weight byte is loaded once with 16-byte streaming loads (L1 bypass),
//     a warp instruction covering 512 contiguous bytes of one row, several rows
//     and vectors per thread in flight;
//   * the activation rows x (fp32: rounding them to BF16 would move 16-layer
//     logits by ~5e-2) sit in shared memory for the whole CTA;
//   * rows are split over CTAs in equal contiguous ranges (the grid is a
//     multiple of the SM count), so every SM streams the same number of bytes;
//     where every CTA owns several 8-row groups, half of each range is fixed
//     and the rest is claimed group by group from an atomic counter, because
//     CTAs do not stream at equal rates and the slowest one sets the time;
//   * FP8-e4m3 weights are converted in registers and the per-output-channel
//     scale is applied once to the finished dot product, which is exact
//     reassociation ("Epilogue and dequant fusion", same section 11);
//   * three epilogues: fp32 partial sums (split-K), the SwiGLU activation over
//     the fused gate/up rows ("Kernels, Fusion & CUDA Graphs", "Fix 1: kernel
//     fusion": gate + up projection and SiLU x mul), and a per-CTA arg-max over
//     LM-head rows so that logits need not reach HBM (same table, "Sampling").
#include "common.cuh"
#include "internal.h"
#include "sampling.cuh"

namespace mbt {

template <int NB> struct GemvShape;
template <> struct GemvShape<1> { static constexpr int RG = 8, U = 2, MINB = 2; };
template <> struct GemvShape<2> { static constexpr int RG = 8, U = 2, MINB = 2; };
template <> struct GemvShape<4> { static constexpr int RG = 4, U = 2, MINB = 2; };
template <> struct GemvShape<8> { static constexpr int RG = 4, U = 2, MINB = 1; };

constexpr int kGemvThreads = 256;
#ifndef MBT_GEMV_PREFETCH_KB
#define MBT_GEMV_PREFETCH_KB 64
#endif
constexpr int kGemvPrefetchKB = MBT_GEMV_PREFETCH_KB;   // default L2 prefetch per CTA before the PDL wait
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

// Four weights of a 16-byte vector (quarter q) widened to fp32, exactly.
template <int WT>
__device__ __forceinline__ void widen4(const uint4& w, int q, float (&f)[4]);

template <>
__device__ __forceinline__ void widen4<W_BF16>(const uint4& w, int q, float (&f)[4]) {
  const uint32_t a = q ? w.z : w.x, b = q ? w.w : w.y;
  f[0] = bf16_lo(a); f[1] = bf16_hi(a); f[2] = bf16_lo(b); f[3] = bf16_hi(b);
}

template <>
__device__ __forceinline__ void widen4<W_E4M3>(const uint4& w, int q, float (&f)[4]) {
  const uint32_t a = q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w;
  const float2 lo = e4m3x2_to_float2(a), hi = e4m3x2_to_float2(a >> 16);
  f[0] = lo.x; f[1] = lo.y; f[2] = hi.x; f[3] = hi.y;
}

template <int NB, int WT, int EPI, int PRO>
__global__ void __launch_bounds__(kGemvThreads, GemvShape<NB>::MINB)
gemv_kernel(const GemvArgs a) {
  constexpr int RG = GemvShape<NB>::RG;          // weight rows per group
  constexpr int U = GemvShape<NB>::U;            // 16-B vectors per row per thread in flight
  constexpr int EPV = (WT == W_BF16) ? 8 : 16;   // elements per 16-B weight vector
  constexpr int QN = EPV / 4;                    // fp32 quarters (float4) of x per vector
  constexpr int M = RG * NB;                     // dot products per group
  constexpr int CH = (EPI == EPI_SWIGLU) ? RG / 2 : RG;   // output channels per group
  static_assert(M <= 32 && (M & (M - 1)) == 0, "M must be a power of two <= 32");

  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();

  // this CTA's split of K, in 16-byte weight vectors
  const int nvec_all = a.K / EPV;
  const int split = blockIdx.y, nsplit = gridDim.y;
  const int v0 = (int)((long long)nvec_all * split / nsplit);
  const int nvec = (int)((long long)nvec_all * (split + 1) / nsplit) - v0;
  const int G = gridDim.x, c = blockIdx.x;
  const int r_begin = (int)((long long)a.N * c / G);
  const int r_end = (int)((long long)a.N * (c + 1) / G);
  const size_t row_bytes = (size_t)a.K * (WT == W_BF16 ? 2 : 1);
  const unsigned char* Wb = reinterpret_cast<const unsigned char*>(a.W) + (size_t)v0 * 16;

  // Static part of the schedule: the CTA's contiguous range of rows, or with a
  // work queue its first static_groups groups (the rest is claimed later).
  int rb = r_begin, re = r_end;
  int* const sched = a.sched ? a.sched + split : nullptr;
  const int dyn0 = a.sched ? G * a.static_groups * CH : a.N;
  if (sched) {
    rb = min(a.N, c * a.static_groups * CH);
    re = min(a.N, rb + a.static_groups * CH);
  }

  // The weights do not depend on the previous kernel: pull this CTA's first
  // rows (all of them when prefetch_bytes says so) into L2 while it drains.
  if (rb < re) {
    const size_t seg = (size_t)nvec * 16;                       // this split's bytes of a row
    const size_t budget = a.prefetch_bytes ? a.prefetch_bytes : (size_t)kGemvPrefetchKB * 1024;
    const int rows = (EPI == EPI_SWIGLU ? 2 : 1) * (re - rb);
    const int n_pf = (int)min((size_t)rows, max((size_t)1, budget / seg));
    for (int i = tid; i < n_pf; i += kGemvThreads) {
      const int ch = rb + (EPI == EPI_SWIGLU ? i / 2 : i);
      const int wr = (EPI == EPI_SWIGLU && (i & 1)) ? a.N + ch : ch;
      const unsigned char* rp = Wb + (size_t)wr * row_bytes;
      for (size_t o = 0; o < seg; o += 65536)
        prefetch_l2(rp + o, (uint32_t)min(seg - o, (size_t)65536));
    }
  }
  // the norm's gain is a weight too: into registers before the wait
  constexpr int kGammaPre = 8;
  uint2 gpre[kGammaPre];
  if (PRO == PRO_NORM) {
#pragma unroll
    for (int j = 0; j < kGammaPre; ++j) {
      const int k4 = tid + j * kGemvThreads;
      gpre[j] = k4 < a.K / 4 ? reinterpret_cast<const uint2*>(a.gamma)[k4] : make_uint2(0u, 0u);
    }
  }
  pdl_wait();

  // x tile (fp32): [NB][QN][nvec] float4, so that a warp reads 512 contiguous bytes
  float4* xs = reinterpret_cast<float4*>(smem);
  const int xrow = nvec * QN;
  float* red = reinterpret_cast<float*>(smem + (size_t)NB * xrow * 16);   // [2][warps][32]
  float* fin = red + 2 * kGemvWarps * 32;                                  // [M]
  if (PRO == PRO_X) {
    // coalesced float4 reads of this split's slice of each row, XU in flight
    // per thread, scattered into the [q][v] layout of the tile
    const float* xb = a.x + (size_t)v0 * EPV;
    constexpr int XU = 8;
    const int k4n = xrow;                                // float4 per row in this split
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const bool live = b < a.nb;
      const float4* __restrict__ x4 = reinterpret_cast<const float4*>(xb + (size_t)b * a.ldx);
      for (int base = 0; base < k4n; base += XU * kGemvThreads) {
        float4 val[XU];
#pragma unroll
        for (int j = 0; j < XU; ++j) {
          const int k4 = base + tid + j * kGemvThreads;
          val[j] = (live && k4 < k4n) ? x4[k4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < XU; ++j) {
          const int k4 = base + tid + j * kGemvThreads;
          if (k4 < k4n) {
            const int vv = k4 / QN, q = k4 - vv * QN;
            xs[(b * QN + q) * nvec + vv] = val[j];
          }
        }
      }
    }
  } else {
    // RMSNorm prologue (nsplit == 1): x = (r_in + sum_s delta_s) / rms * gamma.
    // "Residual add + RMSNorm" ("Kernels, Fusion & CUDA Graphs", "Fix 1: kernel
    // fusion") done by every CTA into its own x tile; CTA 0 stores the new residual.
    const int k4n = a.K / 4;
    const bool store_r = (c == 0 && split == 0);
    constexpr int PV = 4;                        // float4 of r per thread per pass
    constexpr int ND = 3;                        // partials loaded with r in the same round trip
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      ss[b] = 0.f;
      const bool live = b < a.nb;
      const float4* __restrict__ r4 = reinterpret_cast<const float4*>(a.r_in + (size_t)b * a.K);
      const float4* __restrict__ d4 = reinterpret_cast<const float4*>(a.delta + (size_t)b * a.K);
      float4* __restrict__ o4 = reinterpret_cast<float4*>(a.r_out + (size_t)b * a.K);
      const size_t dst4 = (size_t)(a.delta_stride / 4);
      for (int base = 0; base < k4n; base += PV * kGemvThreads) {
        // the loads of r and of the first ND partials first (one round trip),
        // then the sums in the fixed order r + d0 + d1 + ...
        float4 v[PV], t[ND][PV];
#pragma unroll
        for (int j = 0; j < PV; ++j) {
          const int k4 = base + tid + j * kGemvThreads;
          const bool in = live && k4 < k4n;
          v[j] = in ? r4[k4] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int sd = 0; sd < ND; ++sd)
            t[sd][j] = (in && sd < a.n_delta) ? d4[sd * dst4 + k4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int sd = 0; sd < ND; ++sd)
          if (sd < a.n_delta) {
#pragma unroll
            for (int j = 0; j < PV; ++j) {
              v[j].x += t[sd][j].x; v[j].y += t[sd][j].y; v[j].z += t[sd][j].z; v[j].w += t[sd][j].w;
            }
          }
        for (int sidx = ND; sidx < a.n_delta; ++sidx) {
#pragma unroll
          for (int j = 0; j < PV; ++j) {
            const int k4 = base + tid + j * kGemvThreads;
            const float4 u = (live && k4 < k4n) ? d4[sidx * dst4 + k4] : make_float4(0.f, 0.f, 0.f, 0.f);
            v[j].x += u.x; v[j].y += u.y; v[j].z += u.z; v[j].w += u.w;
          }
        }
#pragma unroll
        for (int j = 0; j < PV; ++j) {
          const int k4 = base + tid + j * kGemvThreads;
          if (k4 < k4n) {
            if (store_r && live) o4[k4] = v[j];
            ss[b] += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
            const int vv = k4 / QN, q = k4 - vv * QN;
            xs[(b * QN + q) * nvec + vv] = v[j];
          }
        }
      }
      ss[b] = warp_sum(ss[b]);
    }
    if (lane == 0) {
#pragma unroll
      for (int b = 0; b < NB; ++b) red[warp * NB + b] = ss[b];
    }
    __syncthreads();
    float inv[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float t = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kGemvWarps; ++w2) t += red[w2 * NB + b];
      inv[b] = 1.0f / sqrtf(t / (float)a.K + a.eps);
    }
    const uint2* g2 = reinterpret_cast<const uint2*>(a.gamma);
#pragma unroll 8
    for (int k4 = tid; k4 < k4n; k4 += kGemvThreads) {
      const int j = (k4 - tid) / kGemvThreads;
      const uint2 g = j < kGammaPre ? gpre[j] : g2[k4];
      const float g0 = bf16_lo(g.x), g1 = bf16_hi(g.x), gg2 = bf16_lo(g.y), g3 = bf16_hi(g.y);
      const int v = k4 / QN, q = k4 - v * QN;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float4& x = xs[(b * QN + q) * nvec + v];
        x.x = x.x * inv[b] * g0; x.y = x.y * inv[b] * g1;
        x.z = x.z * inv[b] * gg2; x.w = x.w * inv[b] * g3;
      }
    }
  }
  __syncthreads();

  float best_v = -INFINITY;
  int best_i = 0x7fffffff;
  int buf = 0;
  // Work-queue tail: CTAs stream at unequal rates (a fixed split left the
  // last CTA of a batch-1 gate/up projection ~60% behind the median), so
  // after the static part each CTA claims one group at a time. Thread 0 claims
  // the next group when it starts the last group of its current range, so
  // the atomic's round trip hides behind that group's loads; groups are
  // claimed in increasing order, so every CTA still sees its rows ascending.
  __shared__ int s_next;
  int claim = 0;
  if (sched && tid == 0 && rb >= re) claim = atomicAdd(sched, 1);

  for (;;) {
  for (int r0 = rb; r0 < re; r0 += CH, buf ^= 1) {
    if (sched && tid == 0 && r0 + CH >= re) claim = atomicAdd(sched, 1);
    const unsigned char* rowp[RG];
#pragma unroll
    for (int i = 0; i < RG; ++i) {
      int ch = r0 + (i % CH);
      ch = ch < re ? ch : re - 1;
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
          for (int q = 0; q < QN; ++q) {
            float4 xq[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) xq[b] = xs[(b * QN + q) * nvec + vv];
#pragma unroll
            for (int i = 0; i < RG; ++i) {
              float wf[4];
              widen4<WT>(w[u][i], q, wf);
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                float s = acc[i * NB + b];
                s = fmaf(wf[0], xq[b].x, s);
                s = fmaf(wf[1], xq[b].y, s);
                s = fmaf(wf[2], xq[b].z, s);
                s = fmaf(wf[3], xq[b].w, s);
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
        if (ch < re && b < a.nb) {
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
        if (ch < re && b < a.nb) {
          if (WT == W_E4M3) { g *= a.scale[ch]; u *= a.scale[a.N + ch]; }
          a.act[(size_t)b * a.lda + ch] = g / (1.f + expf(-g)) * u;
        }
      }
    } else {  // EPI_ARGMAX
      if (tid < M) {
        const int i = tid / NB, b = tid % NB, ch = r0 + i;
        float t = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kGemvWarps; ++w2) t += rb[w2 * 32 + tid];
        if (WT == W_E4M3 && ch < re) t *= a.scale[ch];
        fin[tid] = t;
        if (ch < re && b < a.nb && a.logits) a.logits[(size_t)b * a.ldl + ch] = t;
      }
      __syncthreads();
      if (tid < NB) {
#pragma unroll
        for (int i = 0; i < RG; ++i) {
          const int ch = r0 + i;
          if (ch < re) {
            float t = fin[i * NB + tid];
            if (a.gum.on && t == t) t = gumbel_score(t, ch, tid, a.gum);
            if (t > best_v) { best_v = t; best_i = ch; }          // rows ascend: first max kept
            else if (!(t == t)) set_err(a.err, MBT_DEV_NONFINITE);
          }
        }
      }
    }
  }
  if (!sched) break;
  // every thread has read the previous s_next: the range above held at least
  // one group (with its barrier), or this is the first claim
  if (tid == 0) s_next = claim;
  __syncthreads();
  rb = dyn0 + s_next * CH;
  re = min(a.N, rb + CH);
  if (rb >= re) {
    // Every CTA ends with one claim past the last group, so the counter
    // takes n_dyn + grid claims in all; whoever holds the very last one is
    // the last to touch it and leaves it at zero for the next launch.
    const int n_dyn = dyn0 < a.N ? (a.N - dyn0 + CH - 1) / CH : 0;
    if (tid == 0 && s_next == n_dyn + G - 1) atomicExch(sched, 0);
    break;
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
constexpr size_t kXsMax = 216 * 1024;            // largest x tile (1 CTA per SM)
constexpr size_t kXsTwoPerSm = 110 * 1024;       // largest CTA footprint two of which share an SM
// work queue: share of each CTA's groups assigned up front, and the fewest
// groups per CTA for which the queue is used at all
constexpr double kStaticShare = 0.5;
constexpr int kMinGroupsPerCta = 4;

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
void* kernel_ptr(int pro) {
  return pro == PRO_NORM ? (void*)gemv_kernel<NB, WT, EPI, PRO_NORM> : (void*)gemv_kernel<NB, WT, EPI, PRO_X>;
}

void* pick(int nbt, int wt, int epi, int pro) {
#define MBT_PICK_E(NB, WT)                                               \
  switch (epi) {                                                         \
    case EPI_PARTIAL: return kernel_ptr<NB, WT, EPI_PARTIAL>(pro);       \
    case EPI_SWIGLU: return kernel_ptr<NB, WT, EPI_SWIGLU>(pro);         \
    default: return kernel_ptr<NB, WT, EPI_ARGMAX>(pro);                 \
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

int gemv_max_rows(int epi, int K, int pro) {
  if (epi == EPI_PARTIAL && pro == PRO_X) return 8;
  const size_t per_row = (size_t)K * 4;
  for (int nb = 8; nb > 1; nb >>= 1)
    if ((size_t)nb * per_row <= kXsMax) return nb;
  return 1;
}

GemvLaunch gemv_plan(int epi, int wtype, int nb, int N, int K, int num_sms, int force_nsplit, int pro,
                     const StreamCfg& sc) {
  GemvLaunch g;
  const size_t xs_budget = sc.cta_smem - 3 * 1024;     // x tile that still lets 2 CTAs share an SM
  g.nb_tmpl = nb_template(nb);
  const int epv = wtype == W_BF16 ? 8 : 16;
  const int nvec_all = K / epv;
  const size_t xs_full = (size_t)g.nb_tmpl * K * 4;
  int ns = (int)((xs_full + xs_budget - 1) / xs_budget);
  if (g.nb_tmpl == 8) ns = (int)((xs_full + kXsMax - 1) / kXsMax);
  if (epi != EPI_PARTIAL) ns = 1;
  if (force_nsplit > 0) ns = force_nsplit;
  if (pro == PRO_NORM) ns = 1;              // the norm needs the whole row in one CTA
  if (ns > nvec_all) ns = nvec_all;
  if (ns < 1) ns = 1;
  g.nsplit = ns;
  const size_t nvec_max = (size_t)(nvec_all + ns - 1) / ns;
  g.smem = (size_t)g.nb_tmpl * nvec_max * 16 * (epv / 4) + 2 * kGemvWarps * 32 * 4 + 32 * 4;
  // Two CTAs per SM under the step's L1 split when the x tile fits its budget;
  // a larger tile (4 rows of a norm-prologue projection, whose K cannot be
  // split) still runs two per SM, with the driver's default split for that
  // launch; only 8-row tiles run one per SM.
  const bool fits = g.smem <= sc.cta_smem;
  const int per_sm = (g.nb_tmpl < 8 && (fits || g.smem <= kXsTwoPerSm)) ? 2 : 1;
  g.carveout = fits && per_sm == 2 ? sc.carveout : -1;
  int grid = num_sms * per_sm / ns;
  if (grid < 1) grid = 1;
  const int rg = rows_per_group(g.nb_tmpl, epi);
  g.group_rows = rg;
  const int max_grid = (N + rg - 1) / rg;
  if (grid > max_grid) grid = max_grid;
  g.grid = grid;
  return g;
}

StreamCfg stream_config(size_t attn_bytes, int o_k) {
  const size_t kb = 1024;
  const size_t gemv1 = (size_t)o_k * 4 + 2 * kGemvWarps * 32 * 4 + 32 * 4;   // batch-1 O-projection CTA
  const size_t need = attn_bytes + gemv1 + 2 * kb;                             // + 1 KB reserved per CTA
  const int cfgs[5] = {100, 132, 164, 196, 228};
  StreamCfg c;
  for (int kbs : cfgs) {
    if ((size_t)kbs * kb >= need || kbs == 228) {
      c.carveout = (kbs * 100 + 114) / 228;                                    // nearest percent
      c.cta_smem = ((size_t)kbs * kb - 2 * kb) / 2;
      if (c.cta_smem > kXsMax) c.cta_smem = kXsMax;
      break;
    }
  }
  return c;
}

int gemv_queue_static_groups(const GemvLaunch& g, int N) {
  // only where a CTA's share spans several groups: one group of a long row
  // is a sizeable part of the launch, and claiming it late is the tail
  const int ng = (N + g.group_rows - 1) / g.group_rows;
  if (ng < kMinGroupsPerCta * g.grid) return -1;
  return (int)(kStaticShare * ng / g.grid);
}

cudaError_t gemv_launch(int epi, int pro, const GemvArgs& a, const GemvLaunch& g, cudaStream_t s) {
  void* fn = pick(g.nb_tmpl, a.wtype, epi, pro);
  GemvArgs args = a;
  void* params[] = {&args};
  return launch_pdl(fn, dim3(g.grid, g.nsplit), dim3(kGemvThreads), g.smem, s, params, g.carveout);
}

cudaError_t gemv_init() {
  const int nbs[4] = {1, 2, 4, 8};
  for (int i = 0; i < 4; ++i)
    for (int wt = 0; wt < 2; ++wt)
      for (int epi = 0; epi < 3; ++epi)
        for (int pro = 0; pro < 2; ++pro) {
          // 227 KB per CTA in all, static shared memory included
          const void* fn = pick(nbs[i], wt, epi, pro);
          cudaFuncAttributes fa;
          cudaError_t e = cudaFuncGetAttributes(&fa, fn);
          if (e != cudaSuccess) return e;
          const int lim = 227 * 1024 - (int)fa.sharedSizeBytes;
          e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
          if (e != cudaSuccess) return e;
        }
  return cudaSuccess;
}

}  // namespace mbt
