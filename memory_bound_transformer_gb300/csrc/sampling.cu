// Top-k / top-p sampling of the next token from one row of logits per CTA
// ("Kernels, Fusion & CUDA Graphs", "Fix 1: kernel fusion", the "Sampling"
// row: softmax, top-k / top-p, sample).
//
// What it computes, per row: z = logit / T; the k largest z (a tie at the
// boundary keeps the lower token id); softmax over them; the shortest prefix,
// in order of decreasing probability, whose probabilities reach top_p; then
// the Gumbel-max draw over that prefix (the token with the largest
// z + Gumbel(token); sampling.cuh).
//
// How: the k-th largest z is found by a most-significant-digit radix select
// over an order-preserving 32-bit key of the fp32 value (four passes of 8-bit
// digit histograms, integer counts, so the result does not depend on the
// order threads run in); the keys above it and the lowest-id keys equal to it
// are gathered into shared memory; ranking each candidate against all others
// sorts them; a block-wide scan in that order gives the cumulative
// probabilities; an arg-max over the kept prefix takes the draw.
#include "common.cuh"
#include "internal.h"
#include "sampling.cuh"

namespace mbt {

constexpr int kSampleThreads = 1024;
constexpr int kTieCap = 1024;          // keys equal to the k-th largest that are collected

// fp32 -> uint32 whose unsigned order is the float order (NaN excluded).
__device__ __forceinline__ uint32_t order_key(float z) {
  const uint32_t u = __float_as_uint(z);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive block-wide sum scan of one value per thread, in thread order.
__device__ __forceinline__ float block_scan(float v, float* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    warp_tot[lane] = w;                 // inclusive prefix of warp totals
  }
  __syncthreads();
  const float before = warp ? warp_tot[warp - 1] : 0.f;
  __syncthreads();
  return v + before;
}

__global__ void __launch_bounds__(kSampleThreads) sample_topk_kernel(const TopKArgs a) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix, s_need, n_gt, n_eq;
  __shared__ uint32_t c_key[kTopKMax];
  __shared__ int c_id[kTopKMax];
  __shared__ int ties[kTieCap];
  __shared__ int order[kTopKMax];
  __shared__ float warp_tot[32];
  __shared__ float best_v[32];
  __shared__ int best_i[32];

  const int row = blockIdx.x, tid = threadIdx.x;
  const float* z0 = a.logits + (size_t)row * a.ldl;
  const int K = min(a.k, a.V);

  // 1. radix select of the K-th largest key
  uint32_t prefix = 0, mask = 0, need = (uint32_t)K;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < a.V; i += blockDim.x) {
      const float z = z0[i] * a.inv_t;
      if (!(z == z)) continue;
      const uint32_t key = order_key(z);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t above = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (above + hist[d] >= need) break;
        above += hist[d];
      }
      s_prefix = prefix | ((uint32_t)d << shift);
      s_need = need - above;
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    mask |= 255u << shift;
  }
  // prefix: the K-th largest key; `need` keys equal to it complete the top K
  if (tid == 0) { n_gt = 0; n_eq = 0; }
  __syncthreads();

  // 2. gather the keys above it and the ids of keys equal to it
  for (int i = tid; i < a.V; i += blockDim.x) {
    const float z = z0[i] * a.inv_t;
    if (!(z == z)) { set_err(a.err, MBT_DEV_NONFINITE); continue; }
    const uint32_t key = order_key(z);
    if (key > prefix) {
      const uint32_t s = atomicAdd(&n_gt, 1u);
      if (s < (uint32_t)kTopKMax) { c_key[s] = key; c_id[s] = i; }
    } else if (key == prefix) {
      const uint32_t s = atomicAdd(&n_eq, 1u);
      if (s < (uint32_t)kTieCap) ties[s] = i;
    }
  }
  __syncthreads();
  const int ngt = (int)min(n_gt, (uint32_t)kTopKMax);
  const int neq = (int)min(n_eq, (uint32_t)kTieCap);
  // the `need` lowest ids among the equal keys
  for (int t = tid; t < neq; t += blockDim.x) {
    int r = 0;
    for (int j = 0; j < neq; ++j) r += ties[j] < ties[t];
    if (r < (int)need && ngt + r < kTopKMax) { c_key[ngt + r] = prefix; c_id[ngt + r] = ties[t]; }
  }
  __syncthreads();
  const int nc = min(K, ngt + min((int)need, neq));

  // 3. order the candidates: larger key first, lower id first on equal keys
  for (int t = tid; t < nc; t += blockDim.x) {
    int r = 0;
    for (int j = 0; j < nc; ++j)
      r += (c_key[j] > c_key[t]) || (c_key[j] == c_key[t] && c_id[j] < c_id[t]);
    order[r] = t;
  }
  __syncthreads();

  // 4. probabilities in that order and their running sum (one per thread;
  // K <= blockDim.x)
  const float zmax = nc ? z0[c_id[order[0]]] * a.inv_t : 0.f;
  float p = 0.f, logit = -INFINITY;
  int id = 0x7fffffff;
  if (tid < nc) {
    id = c_id[order[tid]];
    logit = z0[id];
    p = expf(logit * a.inv_t - zmax);
  }
  const float csum = block_scan(p, warp_tot);
  __shared__ float s_total;
  if (tid == nc - 1) s_total = csum;
  __syncthreads();
  // kept: the prefix up to and including the first position where the
  // running sum reaches top_p of the total
  const float reach = a.top_p * s_total;
  const bool before_reach = tid < nc && (tid == 0 || (csum - p) < reach);
  const bool kept = a.top_p >= 1.f ? tid < nc : before_reach;

  // 5. Gumbel-max over the kept tokens (exact ties: lower id)
  float v = kept ? gumbel_score(logit, id, row, a.gum) : -INFINITY;
  int vi = kept ? id : 0x7fffffff;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, vi, o);
    if (ov > v || (ov == v && oi < vi)) { v = ov; vi = oi; }
  }
  const int lane = tid & 31, warp = tid >> 5;
  if (lane == 0) { best_v[warp] = v; best_i[warp] = vi; }
  __syncthreads();
  if (warp == 0) {
    v = lane < (int)(blockDim.x >> 5) ? best_v[lane] : -INFINITY;
    vi = lane < (int)(blockDim.x >> 5) ? best_i[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, vi, o);
      if (ov > v || (ov == v && oi < vi)) { v = ov; vi = oi; }
    }
    if (lane == 0) a.next_ids[row] = vi == 0x7fffffff ? 0 : vi;
  }
}

cudaError_t launch_sample_topk(const TopKArgs& a, cudaStream_t s) {
  if (a.k < 1 || a.k > kTopKMax || a.V < 1) return cudaErrorInvalidValue;
  sample_topk_kernel<<<a.B, kSampleThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mbt
