// Small per-row kernels of the decode step: embedding + RMSNorm, fused
// residual add + RMSNorm, RoPE fused with the paged KV-cache write, the final
// arg-max reduction and the staging of caller inputs into graph buffers.
#include "common.cuh"
#include "internal.h"

namespace mbt {

constexpr int kRowThreads = 256;

// RMSNorm ("Root Mean Square Layer Normalization", reference 9 of "Kernel
// Fusion for Large-Scale LLM Inference"): y = r / sqrt(mean(r^2) + eps) * gamma,
// computed in fp32 and rounded once to BF16 for the next projection.
__device__ __forceinline__ void norm_row(const float* r, int H, const bf16* gamma, float eps,
                                         bf16* y, float* scratch) {
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) { const float v = r[i]; ss = fmaf(v, v, ss); }
  const float tot = block_sum(ss, scratch);
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    y[i] = __float2bfloat16_rn(r[i] * inv * __bfloat162float(gamma[i]));
}

__global__ void __launch_bounds__(kRowThreads) embed_rmsnorm_kernel(const EmbedNormArgs a) {
  __shared__ float scratch[32];
  const int b = blockIdx.x;
  int tok = a.tokens[b];
  if (tok < 0 || tok >= a.vocab) {
    if (threadIdx.x == 0) set_err(a.err, MBT_DEV_TOKEN_RANGE);
    tok = 0;
  }
  const bf16* e = a.embed + (size_t)tok * a.H;
  float* r = a.r + (size_t)b * a.H;
  for (int i = threadIdx.x; i < a.H; i += blockDim.x) r[i] = __bfloat162float(e[i]);
  __syncthreads();
  norm_row(r, a.H, a.gamma, a.eps, a.y + (size_t)b * a.H, scratch);
}

// "Residual add + RMSNorm ... doing both in one pass" ("Kernels, Fusion & CUDA
// Graphs", "Fix 1: kernel fusion"). The projection before it left its output
// as split-K partial sums; they are added here too, in a fixed order.
__global__ void __launch_bounds__(kRowThreads) add_rmsnorm_kernel(const AddNormArgs a) {
  __shared__ float scratch[32];
  const int b = blockIdx.x;
  float* r = a.r + (size_t)b * a.H;
  for (int i = threadIdx.x; i < a.H; i += blockDim.x) {
    float v = r[i];
    for (int s = 0; s < a.n_delta; ++s) v += a.delta[(size_t)s * a.delta_stride + (size_t)b * a.H + i];
    r[i] = v;
  }
  __syncthreads();
  norm_row(r, a.H, a.gamma, a.eps, a.y + (size_t)b * a.H, scratch);
}

cudaError_t launch_embed_rmsnorm(const EmbedNormArgs& a, cudaStream_t s) {
  embed_rmsnorm_kernel<<<a.B, kRowThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_add_rmsnorm(const AddNormArgs& a, cudaStream_t s) {
  add_rmsnorm_kernel<<<a.B, kRowThreads, 0, s>>>(a);
  return cudaGetLastError();
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

__global__ void __launch_bounds__(kRowThreads) rope_kv_write_kernel(const RopeKvArgs a) {
  const int b = blockIdx.x;
  const int half = a.d / 2;
  int pos = a.positions[b];
  bool write = true;
  if (pos < 0 || pos >= a.max_pos) {
    if (threadIdx.x == 0) set_err(a.err, MBT_DEV_POS_RANGE);
    pos = 0;
    write = false;
  }
  const int jb = pos / kBlockTokens, slot = pos % kBlockTokens;
  int blk = -1;
  if (write) {
    blk = jb < a.bt_stride ? a.bt[(size_t)b * a.bt_stride + jb] : -1;
    if (blk < 0 || blk > a.num_blocks) {
      if (threadIdx.x == 0) set_err(a.err, MBT_DEV_BLOCK_RANGE);
      write = false;
    }
  }
  const float* src = a.qkv + (size_t)b * a.ld_qkv;
  const float2* cs = a.rope + (size_t)pos * half;
  const int n_rot = (a.nq + a.nkv) * half;
  for (int e = threadIdx.x; e < n_rot; e += blockDim.x) {
    const int hh = e / half, i = e - hh * half;
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
      const int kvh = hh - a.nq;
      const size_t base = (((size_t)blk * a.nkv + kvh) * kBlockTokens + slot) * a.d;
      store_kv(a.kpool, base + i, __fdiv_rn(y1, a.k_scale), a.kv_fp8);
      store_kv(a.kpool, base + i + half, __fdiv_rn(y2, a.k_scale), a.kv_fp8);
    }
  }
  if (!write) return;
  const int n_v = a.nkv * a.d;
  const int vcol0 = (a.nq + a.nkv) * a.d;
  for (int e = threadIdx.x; e < n_v; e += blockDim.x) {
    const int kvh = e / a.d, i = e - kvh * a.d;
    float v = 0.f;
    for (int s = 0; s < a.nsplit; ++s) v += src[(size_t)s * a.split_stride + vcol0 + e];
    const size_t base = (((size_t)blk * a.nkv + kvh) * kBlockTokens + slot) * a.d;
    store_kv(a.vpool, base + i, __fdiv_rn(v, a.v_scale), a.kv_fp8);
  }
}

cudaError_t launch_rope_kv_write(const RopeKvArgs& a, cudaStream_t s) {
  rope_kv_write_kernel<<<a.B, kRowThreads, 0, s>>>(a);
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
                                 int* next_ids, uint32_t* err, cudaStream_t s) {
  (void)err;
  argmax_reduce_kernel<<<B, kRowThreads, 0, s>>>(part, part_ld, G, next_ids);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Static input buffers for graph replay ("copies inputs into the graph's static
// buffers", "Kernels, Fusion & CUDA Graphs", "Fix 2: CUDA graphs"): rows [B, R)
// become padding rows (token 0, position 0, one token of context in the null
// block) whose only write is to the null block.

__global__ void stage_inputs_kernel(const StageArgs a) {
  const int b = blockIdx.x;
  const bool live = b < a.B;
  if (threadIdx.x == 0) {
    a.s_tok[b] = live ? a.tok[b] : 0;
    a.s_pos[b] = live ? a.pos[b] : 0;
    a.s_sl[b] = live ? a.sl[b] : 1;
  }
  for (int j = threadIdx.x; j < a.s_stride; j += blockDim.x) {
    int v = a.null_block;
    if (live && j < a.bt_stride) v = a.bt[(size_t)b * a.bt_stride + j];
    a.s_bt[(size_t)b * a.s_stride + j] = v;
  }
}

cudaError_t launch_stage_inputs(const StageArgs& a, cudaStream_t s) {
  stage_inputs_kernel<<<a.R, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mbt
