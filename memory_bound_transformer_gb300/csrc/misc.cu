// Small per-row kernels of the decode step: embedding + RMSNorm, fused
// residual add + RMSNorm, RoPE fused with the paged KV-cache write, the final
// arg-max reduction and the staging of caller inputs into graph buffers.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mbt {

constexpr int kRowThreads = 256;
constexpr int kNormMaxV = 8;        // float4 per thread: H <= 8 * 4 * 1024

cudaError_t launch_ex(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args,
                      bool pdl, int carveout, int cluster_x) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  int n = 0;
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (carveout >= 0) {
    attr[n].id = cudaLaunchAttributePreferredSharedMemoryCarveout;
    attr[n].val.sharedMemCarveout = (unsigned)carveout;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// RMSNorm ("Root Mean Square Layer Normalization", reference 9 of "Kernel
// Fusion for Large-Scale LLM Inference"): y = r / sqrt(mean(r^2) + eps) * gamma,
// in fp32. One CTA per row; every thread keeps its slice of the row in
// registers so the row is read once and written once.
__device__ __forceinline__ void norm_store(const float4 (&v)[kNormMaxV], float ss, int H,
                                          const bf16* __restrict__ gamma, float eps,
                                          float* __restrict__ y, float* scratch) {
  const float tot = block_sum(ss, scratch);
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  const int nv = H / 4;
  const uint2* g2 = reinterpret_cast<const uint2*>(gamma);
  float4* y4 = reinterpret_cast<float4*>(y);
#pragma unroll
  for (int j = 0; j < kNormMaxV; ++j) {
    const int i = threadIdx.x + j * blockDim.x;
    if (i < nv) {
      const uint2 g = g2[i];
      float4 o;
      o.x = v[j].x * inv * bf16_lo(g.x);
      o.y = v[j].y * inv * bf16_hi(g.x);
      o.z = v[j].z * inv * bf16_lo(g.y);
      o.w = v[j].w * inv * bf16_hi(g.y);
      y4[i] = o;
    }
  }
}

__global__ void __launch_bounds__(1024) embed_rmsnorm_kernel(const EmbedNormArgs a) {
  __shared__ float scratch[32];
  const int b = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  // every kernel of the previous step has finished (each waited on its
  // predecessor), and this step's projections start after this kernel
  if (b == 0)
    for (int i = threadIdx.x; i < a.n_zero; i += blockDim.x) a.zero[i] = 0;
  int tok = a.tokens[b];
  if (tok < 0 || tok >= a.vocab) {
    if (threadIdx.x == 0) set_err(a.err, MBT_DEV_TOKEN_RANGE);
    tok = 0;
  }
  const uint2* e = reinterpret_cast<const uint2*>(a.embed + (size_t)tok * a.H);
  float4* r = reinterpret_cast<float4*>(a.r + (size_t)b * a.H);
  const int nv = a.H / 4;
  float4 v[kNormMaxV];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kNormMaxV; ++j) {
    const int i = threadIdx.x + j * blockDim.x;
    if (i < nv) {
      const uint2 u = e[i];
      v[j] = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
      r[i] = v[j];
      ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    }
  }
  if (a.y) norm_store(v, ss, a.H, a.gamma, a.eps, a.y + (size_t)b * a.H, scratch);
}

// "Residual add + RMSNorm ... doing both in one pass" ("Kernels, Fusion & CUDA
// Graphs", "Fix 1: kernel fusion"). The projection before it left its output
// as split-K partial sums; they are added here too, in a fixed order.
// y as 16-bit high/low rows (BF16: y = hi + lo to ~2^-17; FP16 for e4m3
// weights) for the tensor-core GEMM.
__device__ __forceinline__ void norm_store_hl(const float4 (&v)[kNormMaxV], float ss, int H,
                                             const bf16* __restrict__ gamma, float eps, uint16_t* hi_row,
                                             uint16_t* lo_row, float* scratch, int f16) {
  const float tot = block_sum(ss, scratch);
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  const int nv = H / 4;
  const uint2* g2 = reinterpret_cast<const uint2*>(gamma);
#pragma unroll
  for (int j = 0; j < kNormMaxV; ++j) {
    const int i = threadIdx.x + j * blockDim.x;
    if (i < nv) {
      const uint2 g = g2[i];
      const float o[4] = {v[j].x * inv * bf16_lo(g.x), v[j].y * inv * bf16_hi(g.x),
                          v[j].z * inv * bf16_lo(g.y), v[j].w * inv * bf16_hi(g.y)};
#pragma unroll
      for (int e = 0; e < 4; ++e) store_hl16(hi_row + 4 * i + e, lo_row + 4 * i + e, o[e], f16);
    }
  }
}

__global__ void __launch_bounds__(1024) add_rmsnorm_kernel(const AddNormArgs a) {
  __shared__ float scratch[32];
  const int b = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  if (b >= a.B) {                                   // padding rows of the high/low output
    const bf16 z = __float2bfloat16_rn(0.f);
    for (int i = threadIdx.x; i < a.H; i += blockDim.x) {
      a.y_hl[(size_t)b * a.H + i] = z;
      a.y_hl[(size_t)(a.rp + b) * a.H + i] = z;
    }
    return;
  }
  const int nv = a.H / 4;
  float4* __restrict__ r = reinterpret_cast<float4*>(a.r + (size_t)b * a.H);
  const float4* __restrict__ d = reinterpret_cast<const float4*>(a.delta + (size_t)b * a.H);
  const size_t ds = (size_t)a.delta_stride / 4;
  float4 v[kNormMaxV];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kNormMaxV; ++j) {
    const int i = threadIdx.x + j * blockDim.x;
    if (i < nv) {
      float4 x = r[i];
      for (int s = 0; s < a.n_delta; ++s) {
        const float4 t = d[s * ds + i];
        x.x += t.x; x.y += t.y; x.z += t.z; x.w += t.w;
      }
      v[j] = x;
      ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
    }
  }
#pragma unroll
  for (int j = 0; j < kNormMaxV; ++j) {
    const int i = threadIdx.x + j * blockDim.x;
    if (i < nv) r[i] = v[j];
  }
  if (a.y_hl) {
    uint16_t* hl = reinterpret_cast<uint16_t*>(a.y_hl);
    norm_store_hl(v, ss, a.H, a.gamma, a.eps, hl + (size_t)b * a.H, hl + (size_t)(a.rp + b) * a.H, scratch, a.hl_f16);
  }
  else
    norm_store(v, ss, a.H, a.gamma, a.eps, a.y + (size_t)b * a.H, scratch);
}

// The same residual add + RMSNorm with y as four e4m3 term rows and the row's
// power-of-two scale (split_terms), for e4m3 weights. It needs a second pass
// over the row (its largest |y|) and the split, so a row is spread over a
// cluster of C CTAs (one float4 of the row per thread where the row allows
// it): a row per CTA left most SMs idle at batch 32-64 and took ~10 us. The
// CTAs exchange their partial sums of squares, then their largest |y|,
// through distributed shared memory, each in the same fixed order. (For the
// 16-bit outputs the one-CTA-per-row kernel above measured faster inside the
// replayed step: 4.34 against 4.80 ms at 8B batch 16.)
constexpr int kNormThreads = 256;
constexpr int kNormG = 4;          // float4 per thread: H <= 8 CTAs x 256 threads x 4 x 4

__global__ void __launch_bounds__(kNormThreads) add_rmsnorm_terms_kernel(const AddNormArgs a) {
  __shared__ float scratch[32];
  __shared__ float part[2];        // this CTA's sum of squares, largest |y|
  const int C = gridDim.x, c = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  const int nv = a.H / 4, per = (nv + C - 1) / C, i0 = c * per, i1 = min(nv, i0 + per);
  if (b >= a.B) {                  // padding rows: zero codes, scale 1 (the whole cluster)
    for (int i = i0 + tid; i < i1; i += kNormThreads)
      for (int tj = 0; tj < kTerms; ++tj)
        reinterpret_cast<uint32_t*>(a.y_t + ((size_t)tj * a.rp + b) * a.H)[i] = 0u;
    if (c == 0 && tid == 0) a.y_s[b] = 1.f;
    return;
  }
  float4* __restrict__ r = reinterpret_cast<float4*>(a.r + (size_t)b * a.H);
  const float4* __restrict__ d = reinterpret_cast<const float4*>(a.delta + (size_t)b * a.H);
  const size_t ds = (size_t)a.delta_stride / 4;
  float4 v[kNormG];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kNormG; ++j) {
    const int i = i0 + tid + j * kNormThreads;
    if (i < i1) {
      float4 x = r[i];
      for (int s = 0; s < a.n_delta; ++s) {
        const float4 t = d[s * ds + i];
        x.x += t.x; x.y += t.y; x.z += t.z; x.w += t.w;
      }
      v[j] = x;
      r[i] = x;
      ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
    }
  }
  float tot = block_sum(ss, scratch);
  if (C > 1) {
    if (tid == 0) part[0] = tot;
    cluster_sync_all();
    tot = 0.f;
    for (int q = 0; q < C; ++q) tot += ld_dsmem_f32(&part[0], (uint32_t)q);
  }
  const float inv = 1.0f / sqrtf(tot / (float)a.H + a.eps);
  const uint2* g2 = reinterpret_cast<const uint2*>(a.gamma);
  float o[kNormG][4];
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < kNormG; ++j) {
    const int i = i0 + tid + j * kNormThreads;
    if (i < i1) {
      const uint2 g = g2[i];
      o[j][0] = v[j].x * inv * bf16_lo(g.x); o[j][1] = v[j].y * inv * bf16_hi(g.x);
      o[j][2] = v[j].z * inv * bf16_lo(g.y); o[j][3] = v[j].w * inv * bf16_hi(g.y);
#pragma unroll
      for (int e = 0; e < 4; ++e) m = fmaxf(m, fabsf(o[j][e]));
    }
  }
  m = block_max(m, scratch);
  if (C > 1) {
    if (tid == 0) part[1] = m;
    cluster_sync_all();
    m = 0.f;
    for (int q = 0; q < C; ++q) m = fmaxf(m, ld_dsmem_f32(&part[1], (uint32_t)q));
  }
  float sc, isc;
  term_scale(m, sc, isc);
  if (c == 0 && tid == 0) a.y_s[b] = sc;
#pragma unroll
  for (int j = 0; j < kNormG; ++j) {
    const int i = i0 + tid + j * kNormThreads;
    if (i < i1) {
      uint32_t cd[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) cd[e] = split_terms(o[j][e], isc);
#pragma unroll
      for (int tj = 0; tj < kTerms; ++tj) {
        const uint32_t w = ((cd[0] >> (8 * tj)) & 255u) | (((cd[1] >> (8 * tj)) & 255u) << 8) |
                           (((cd[2] >> (8 * tj)) & 255u) << 16) | (((cd[3] >> (8 * tj)) & 255u) << 24);
        reinterpret_cast<uint32_t*>(a.y_t + ((size_t)tj * a.rp + b) * a.H)[i] = w;
      }
    }
  }
  if (C > 1) cluster_sync_all();   // no CTA leaves while the others may still read its partials
}

// One float4 per thread where the row allows it, so a CTA has the whole row
// (and its split-K partials) in flight at once.
static int norm_threads(int H) {
  int t = H / 4;
  t = ((t + 31) / 32) * 32;
  if (t < 128) t = 128;
  if (t > 1024) t = 1024;
  return t;
}

cudaError_t launch_embed_rmsnorm(const EmbedNormArgs& a, cudaStream_t s) {
  if (a.H % 4 || a.H > 4 * kNormMaxV * 1024) return cudaErrorInvalidValue;
  // An ordinary launch: the step's first kernel starts only once everything
  // before it on the stream (the previous step included) has finished, which
  // is what lets later kernels of the step read the step inputs and the KV
  // cache before their programmatic wait.
  EmbedNormArgs args = a;
  void* p[] = {&args};
  return launch_ex((const void*)embed_rmsnorm_kernel, dim3(a.B), dim3(norm_threads(a.H)), 0, s, p, false,
                   a.carveout > 0 ? a.carveout : -1);
}

cudaError_t launch_add_rmsnorm(const AddNormArgs& a, cudaStream_t s) {
  AddNormArgs args = a;
  void* p[] = {&args};
  if (a.y_t) {
    const int nv = a.H / 4;
    const int C = std::min(8, (nv + kNormThreads - 1) / kNormThreads);
    if (a.H % 4 || a.H < 4 || (nv + C - 1) / C > kNormThreads * kNormG || !a.y_s || a.y_hl)
      return cudaErrorInvalidValue;
    return launch_ex((const void*)add_rmsnorm_terms_kernel, dim3(C, a.rp), dim3(kNormThreads), 0, s, p, true, -1,
                     C > 1 ? C : 0);
  }
  if (a.H % 4 || a.H > 4 * kNormMaxV * 1024 || (!a.y_hl && !a.y)) return cudaErrorInvalidValue;
  const int rows = a.y_hl ? a.rp : a.B;
  return launch_pdl((const void*)add_rmsnorm_kernel, dim3(rows), dim3(norm_threads(a.H)), 0, s, p);
}

// ---------------------------------------------------------------------------
// "RoPE + KV-cache write: rotate, then copy into paged blocks ... One read, one
// write" ("Kernels, Fusion & CUDA Graphs", "Fix 1: kernel fusion").
// Rotate-half pairing: element i pairs with i + d/2 and turns by
// pos * theta^(-2i/d) (table built on the host in double precision).
// Token at position p goes to block bt[p / 16], slot p % 16.

__device__ __forceinline__ void store_kv(void* pool, size_t idx, float v, int fp8) {
  if (fp8) reinterpret_cast<uint8_t*>(pool)[idx] = f32_to_e4m3(v);
  else reinterpret_cast<uint16_t*>(pool)[idx] = f32_to_bf16_bits(v);
}

constexpr int kRopeHeads = 4;      // heads per CTA (q, k or v heads)

__global__ void __launch_bounds__(128) rope_kv_write_kernel(const RopeKvArgs a) {
  const int b = blockIdx.y;
  const int half = a.d / 2;
  const int nh = a.nq + 2 * a.nkv;
  int pos = a.positions[b];
  bool write = true;
  if (pos < 0 || pos >= a.max_pos) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_err(a.err, MBT_DEV_POS_RANGE);
    pos = 0;
    write = false;
  }
  const int jb = pos / kBlockTokens, slot = pos % kBlockTokens;
  int blk = -1;
  if (write) {
    blk = jb < a.bt_stride ? a.bt[(size_t)b * a.bt_stride + jb] : -1;
    if (blk < 0 || blk > a.num_blocks) {
      if (threadIdx.x == 0 && blockIdx.x == 0) set_err(a.err, MBT_DEV_BLOCK_RANGE);
      write = false;
    }
  }
  const float* __restrict__ src = a.qkv + (size_t)b * a.ld_qkv;
  const float2* __restrict__ cs = a.rope + (size_t)pos * half;
  const int h0 = blockIdx.x * kRopeHeads;
  for (int e = threadIdx.x; e < kRopeHeads * a.d; e += blockDim.x) {
    const int hh = h0 + e / a.d, i = e % a.d;
    if (hh >= nh) continue;
    if (hh < a.nq + a.nkv) {                       // q or k head: rotate pair (i, i + d/2)
      if (i >= half) continue;
      const int col = hh * a.d + i;
      float x1 = 0.f, x2 = 0.f;
      for (int s = 0; s < a.nsplit; ++s) {
        x1 += src[(size_t)s * a.split_stride + col];
        x2 += src[(size_t)s * a.split_stride + col + half];
      }
      const float2 t = cs[i];
      const float y1 = x1 * t.x - x2 * t.y;
      const float y2 = x2 * t.x + x1 * t.y;
      if (hh < a.nq) {
        float* q = a.q_out + ((size_t)b * a.nq + hh) * a.d;
        q[i] = y1;
        q[i + half] = y2;
      } else if (write) {
        const size_t base = (((size_t)blk * a.nkv + (hh - a.nq)) * kBlockTokens + slot) * a.d;
        store_kv(a.kpool, base + i, __fdiv_rn(y1, a.k_scale), a.kv_fp8);
        store_kv(a.kpool, base + i + half, __fdiv_rn(y2, a.k_scale), a.kv_fp8);
      }
    } else if (write) {                            // v head: copy
      const int kvh = hh - a.nq - a.nkv;
      float v = 0.f;
      for (int s = 0; s < a.nsplit; ++s) v += src[(size_t)s * a.split_stride + hh * a.d + i];
      const size_t base = (((size_t)blk * a.nkv + kvh) * kBlockTokens + slot) * a.d;
      store_kv(a.vpool, base + i, __fdiv_rn(v, a.v_scale), a.kv_fp8);
    }
  }
}

cudaError_t launch_rope_kv_write(const RopeKvArgs& a, cudaStream_t s) {
  const int nh = a.nq + 2 * a.nkv;
  rope_kv_write_kernel<<<dim3((nh + kRopeHeads - 1) / kRopeHeads, a.B), 128, 0, s>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Greedy sampling, second half: the LM-head kernel left one (max, index) per
// CTA and row; pick the best, lowest index on ties.

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(kRowThreads) argmax_reduce_kernel(
    const ArgmaxPart* part, int part_ld, int G, int* next_ids) {
  __shared__ float sv[32];
  __shared__ int si[32];
  const int b = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    const ArgmaxPart p = part[(size_t)g * part_ld + b];
    if (better(p.v, p.i, bv, bi)) { bv = p.v; bi = p.i; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    bv = lane < nw ? sv[lane] : -INFINITY;
    bi = lane < nw ? si[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) next_ids[b] = bi == 0x7fffffff ? 0 : bi;
  }
}

cudaError_t launch_argmax_reduce(int B, const ArgmaxPart* part, int part_ld, int G,
                                 int* next_ids, uint32_t* err, cudaStream_t s, int carveout) {
  (void)err;
  void* p[] = {&part, &part_ld, &G, &next_ids};
  return launch_pdl((const void*)argmax_reduce_kernel, dim3(B), dim3(kRowThreads), 0, s, p, carveout);
}

// ---------------------------------------------------------------------------
// Static input buffers for graph replay ("copies inputs into the graph's static
// buffers", "Kernels, Fusion & CUDA Graphs", "Fix 2: CUDA graphs"): rows [B, R)
// become padding rows (token 0, position 0, one token of context in the null
// block) whose only write is to the null block. A live row's table keeps the
// caller's width: the graph's wider static table is filled with -1 past it
// (never the null block, which would make the graph attend over padding), and
// a seq_len the caller's table cannot hold becomes 0 (flagged), which the
// attention kernel treats exactly as the eager path treats the original.

__global__ void stage_inputs_kernel(const StageArgs a) {
  const int b = blockIdx.x;
  const bool live = b < a.B;
  if (threadIdx.x == 0) {
    a.s_tok[b] = live ? a.tok[b] : 0;
    a.s_pos[b] = live ? a.pos[b] : 0;
    int sl = 1;
    if (live) {
      sl = a.sl[b];
      if (sl > a.bt_stride * kBlockTokens) {
        set_err(a.err, MBT_DEV_SEQLEN_RANGE);
        sl = 0;
      }
    }
    a.s_sl[b] = sl;
  }
  for (int j = threadIdx.x; j < a.s_stride; j += blockDim.x) {
    int v = a.null_block;
    if (live) v = j < a.bt_stride ? a.bt[(size_t)b * a.bt_stride + j] : -1;
    a.s_bt[(size_t)b * a.s_stride + j] = v;
  }
}

cudaError_t launch_stage_inputs(const StageArgs& a, cudaStream_t s) {
  stage_inputs_kernel<<<a.R, 128, 0, s>>>(a);
  return cudaGetLastError();
}

__global__ void stage_prefill_kernel(const PrefillStageArgs a) {
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    a.s_tok[b] = a.tokens[b];
    a.s_pos[b] = a.p0 + b;
    a.s_sl[b] = a.p0 + b + 1;
  }
  for (int j = threadIdx.x; j < a.bt_len; j += blockDim.x) a.s_bt[(size_t)b * a.bt_len + j] = a.bt[j];
}

cudaError_t launch_stage_prefill(const PrefillStageArgs& a, cudaStream_t s) {
  stage_prefill_kernel<<<a.R, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mbt
