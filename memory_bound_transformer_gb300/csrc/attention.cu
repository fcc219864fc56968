// Split-K paged decode attention with grouped-query head sharing.
//
// What it computes: for each query head h of row b,
//   o_h = sum_t softmax_t(q_h . K_t / sqrt(d)) V_t   over t < seq_len[b],
// with K_t, V_t gathered from the paged cache through the block table and the
// KV head shared by the nq/nkv query heads of its group ("GPU Inference
// Internals", "The KV-Cache Ledger": grouped-query attention; "Kernel Fusion for
// Large-Scale LLM Inference", section 11: PagedAttention).
//
// How: FlashAttention-style ("GPU Inference Internals", "Kernels: FlashAttention
// and the Memory Hierarchy": tile K and V into on-chip memory, softmax computed
// incrementally, no score matrix in HBM). One CTA per (split of the context,
// KV head, row) so that a batch-1 step still spreads the KV stream over all SMs;
// each CTA reads its KV blocks once for all query heads of the group, keeps a
// running max and sum per head and writes an unnormalised partial. The last
// CTA of a (row, KV head) to finish -- found with an atomic ticket, nothing
// waits -- merges that group's splits.
#include "common.cuh"
#include "internal.h"

namespace mbt {

constexpr int kAttnThreads = 128;
constexpr int kAttnTile = 64;      // tokens per shared-memory tile (4 blocks)
constexpr int kMaxGroup = 16;      // query heads per KV head

__device__ __forceinline__ void cp_async16(void* s, const void* g) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(s);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

template <int D, int KV8>
struct AttnShape {
  static constexpr int ESZ = KV8 ? 1 : 2;
  static constexpr int ROWB = D * ESZ;               // bytes of one token's K (or V) for one head
  static constexpr int NCH = ROWB / 16;              // 16-byte chunks per row
  static constexpr int EPC = 16 / ESZ;               // elements per chunk
  static constexpr int SWZ = NCH >= 8 ? 7 : NCH - 1; // XOR swizzle of K chunks (bank spread)
  static constexpr int DC = D / 4;                   // 4-element output chunks per head
  static constexpr int HL = kAttnThreads / DC;       // head lanes in the PV phase
  static constexpr int HPT_PV = (kMaxGroup + HL - 1) / HL;
  static constexpr int HPT_QK = kMaxGroup / 2;
  static constexpr size_t SMEM = (size_t)kMaxGroup * D * 4 + 4 * (size_t)kAttnTile * ROWB +
                                 (size_t)kMaxGroup * kAttnTile * 4 + 3 * kMaxGroup * 4;
};

template <int KV8>
__device__ __forceinline__ void chunk_to_float(const uint4& c, float* f);
template <>
__device__ __forceinline__ void chunk_to_float<0>(const uint4& c, float* f) {
  f[0] = bf16_lo(c.x); f[1] = bf16_hi(c.x); f[2] = bf16_lo(c.y); f[3] = bf16_hi(c.y);
  f[4] = bf16_lo(c.z); f[5] = bf16_hi(c.z); f[6] = bf16_lo(c.w); f[7] = bf16_hi(c.w);
}
template <>
__device__ __forceinline__ void chunk_to_float<1>(const uint4& c, float* f) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 a = e4m3x2_to_float2(w[i]), b = e4m3x2_to_float2(w[i] >> 16);
    f[4 * i] = a.x; f[4 * i + 1] = a.y; f[4 * i + 2] = b.x; f[4 * i + 3] = b.y;
  }
}

// One split of one (row, KV head): stream its KV blocks once for all query
// heads of the group and leave (unnormalised o, running max m, sum l) per head.
template <int D, int KV8>
__device__ __forceinline__ void attend(const AttnArgs& a, unsigned char* smem, int b, int h, int sp,
                                       int G, size_t head0, int seq, int blk0, int blk1) {
  using S = AttnShape<D, KV8>;
  float* qs = reinterpret_cast<float*>(smem);                        // [group][D]
  unsigned char* kt = smem + (size_t)kMaxGroup * D * 4;               // [2][tile][ROWB] swizzled
  unsigned char* vt = kt + 2 * (size_t)kAttnTile * S::ROWB;           // [2][tile][ROWB]
  float* sc = reinterpret_cast<float*>(vt + 2 * (size_t)kAttnTile * S::ROWB);   // [group][tile]
  float* st_m = sc + kMaxGroup * kAttnTile;
  float* st_l = st_m + kMaxGroup;
  float* st_a = st_l + kMaxGroup;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // queries of the group, pre-scaled into the log2 domain with the K dequant scale
  const float qscale = 1.4426950408889634f / sqrtf((float)D) * a.k_scale;
  if (a.qkv) {
    // RoPE (rotate-half: element i pairs with i + D/2) straight from the QKV
    // projection's partial sums
    const int half = D / 2;
    int pos = a.positions[b];
    if (pos < 0 || pos >= a.max_pos) pos = 0;
    const float* src = a.qkv + (size_t)b * a.ld_qkv + (size_t)h * G * D;
    const float2* cs = a.rope + (size_t)pos * half;
    for (int e = tid; e < G * half; e += kAttnThreads) {
      const int g = e / half, i = e - g * half;
      float x1 = 0.f, x2 = 0.f;
      for (int s2 = 0; s2 < a.qkv_nsplit; ++s2) {
        x1 += src[(size_t)s2 * a.qkv_split_stride + g * D + i];
        x2 += src[(size_t)s2 * a.qkv_split_stride + g * D + i + half];
      }
      const float2 t = cs[i];
      qs[g * D + i] = (x1 * t.x - x2 * t.y) * qscale;
      qs[g * D + i + half] = (x2 * t.x + x1 * t.y) * qscale;
    }
  } else {
    for (int i = tid; i < G * D; i += kAttnThreads) qs[i] = a.q[head0 * D + i] * qscale;
  }
  if (tid < G) { st_m[tid] = -INFINITY; st_l[tid] = 0.f; }

  const unsigned char* kpool = reinterpret_cast<const unsigned char*>(a.kpool);
  const unsigned char* vpool = reinterpret_cast<const unsigned char*>(a.vpool);
  const int* bt = a.bt + (size_t)b * a.bt_stride;
  const int tok_begin = blk0 * kBlockTokens;
  const int tok_end_blk = blk1 * kBlockTokens;                       // whole blocks loaded
  const int ntiles = (tok_end_blk - tok_begin + kAttnTile - 1) / kAttnTile;

  auto load_tile = [&](int t, int buf) {
    const int tok0 = tok_begin + t * kAttnTile;
    const int rows = min(kAttnTile, tok_end_blk - tok0);
    unsigned char* kd = kt + (size_t)buf * kAttnTile * S::ROWB;
    unsigned char* vd = vt + (size_t)buf * kAttnTile * S::ROWB;
    for (int i = tid; i < rows * S::NCH; i += kAttnThreads) {
      const int row = i / S::NCH, ch = i - row * S::NCH;
      const int tok = tok0 + row;
      int blk = bt[tok / kBlockTokens];
      if (blk < 0 || blk > a.num_blocks) {
        set_err(a.err, MBT_DEV_BLOCK_RANGE);
        blk = a.num_blocks;
      }
      const size_t off = (((size_t)blk * a.nkv + h) * kBlockTokens + (tok % kBlockTokens)) * S::ROWB + ch * 16;
      cp_async16(kd + row * S::ROWB + ((ch ^ (row & S::SWZ)) * 16), kpool + off);
      cp_async16(vd + row * S::ROWB + ch * 16, vpool + off);
    }
    cp_async_commit();
  };

  float o[S::HPT_PV][4];
#pragma unroll
  for (int j = 0; j < S::HPT_PV; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[j][e] = 0.f;
  const int dc = tid % S::DC, hl = tid / S::DC;

  load_tile(0, 0);
  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1;
    if (t + 1 < ntiles) { load_tile(t + 1, buf ^ 1); cp_async_wait<1>(); }
    else cp_async_wait<0>();
    __syncthreads();
    const int tok0 = tok_begin + t * kAttnTile;
    const int nvalid = min(kAttnTile, min(seq, tok_end_blk) - tok0);   // this split's tokens only

    // scores: thread = (token, head parity)
    {
      const int tt = tid & (kAttnTile - 1), hp = tid >> 6;
      float s[S::HPT_QK];
#pragma unroll
      for (int j = 0; j < S::HPT_QK; ++j) s[j] = 0.f;
      const unsigned char* krow = kt + (size_t)buf * kAttnTile * S::ROWB + tt * S::ROWB;
#pragma unroll 4
      for (int ch = 0; ch < S::NCH; ++ch) {
        const uint4 kc = *reinterpret_cast<const uint4*>(krow + ((ch ^ (tt & S::SWZ)) * 16));
        float kf[S::EPC];
        chunk_to_float<KV8>(kc, kf);
#pragma unroll
        for (int j = 0; j < S::HPT_QK; ++j) {
          const int g = hp + 2 * j;
          if (g < G) {
            const float* qg = qs + g * D + ch * S::EPC;
#pragma unroll
            for (int e = 0; e < S::EPC; ++e) s[j] = fmaf(qg[e], kf[e], s[j]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < S::HPT_QK; ++j) {
        const int g = hp + 2 * j;
        if (g < G) sc[g * kAttnTile + tt] = tt < nvalid ? s[j] : -INFINITY;
      }
    }
    __syncthreads();

    // online softmax statistics, one warp per head
    for (int g = warp; g < G; g += kAttnThreads / 32) {
      const float v0 = sc[g * kAttnTile + lane], v1 = sc[g * kAttnTile + lane + 32];
      const float mx = warp_max(fmaxf(v0, v1));
      const float m_old = st_m[g];
      const float m_new = fmaxf(m_old, mx);
      const float p0 = exp2f(v0 - m_new), p1 = exp2f(v1 - m_new);
      sc[g * kAttnTile + lane] = p0;
      sc[g * kAttnTile + lane + 32] = p1;
      const float ps = warp_sum(p0 + p1);
      if (lane == 0) {
        const float al = exp2f(m_old - m_new);
        st_a[g] = al;
        st_l[g] = st_l[g] * al + ps;
        st_m[g] = m_new;
      }
    }
    __syncthreads();

    // o <- o * alpha + P V: thread = (4-element chunk of d, head lane)
    {
#pragma unroll
      for (int j = 0; j < S::HPT_PV; ++j) {
        const int g = hl + S::HL * j;
        if (g < G) {
          const float al = st_a[g];
#pragma unroll
          for (int e = 0; e < 4; ++e) o[j][e] *= al;
        }
      }
      const unsigned char* vb = vt + (size_t)buf * kAttnTile * S::ROWB + dc * 4 * S::ESZ;
      for (int tt = 0; tt < nvalid; ++tt) {
        float vf[4];
        if (KV8) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(vb + tt * S::ROWB);
          const float2 x = e4m3x2_to_float2(w), y = e4m3x2_to_float2(w >> 16);
          vf[0] = x.x; vf[1] = x.y; vf[2] = y.x; vf[3] = y.y;
        } else {
          const uint2 w = *reinterpret_cast<const uint2*>(vb + tt * S::ROWB);
          vf[0] = bf16_lo(w.x); vf[1] = bf16_hi(w.x); vf[2] = bf16_lo(w.y); vf[3] = bf16_hi(w.y);
        }
#pragma unroll
        for (int j = 0; j < S::HPT_PV; ++j) {
          const int g = hl + S::HL * j;
          if (g < G) {
            const float p = sc[g * kAttnTile + tt];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[j][e] = fmaf(p, vf[e], o[j][e]);
          }
        }
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int j = 0; j < S::HPT_PV; ++j) {
    const int g = hl + S::HL * j;
    if (g < G) {
      float4 v = make_float4(o[j][0], o[j][1], o[j][2], o[j][3]);
      *reinterpret_cast<float4*>(a.part_o + ((head0 + g) * a.nsplit + sp) * D + dc * 4) = v;
    }
  }
  if (tid < G) a.part_ml[(head0 + tid) * a.nsplit + sp] = make_float2(st_m[tid], st_l[tid]);
}

// Merge the splits of the group's G query heads: rescale each partial to the
// common maximum, sum, divide by the total softmax mass, apply the V scale.
// One warp per head finds the maximum and the mass; every thread then sums one
// output element over the splits with several loads in flight.
__device__ __forceinline__ void merge_splits(const AttnArgs& a, float* wsm, int G, size_t head0, int D) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ns = a.nsplit;
  for (int g = warp; g < G; g += kAttnThreads / 32) {
    const float2* ml = a.part_ml + (head0 + g) * ns;
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) if (ml[s].y > 0.f) M = fmaxf(M, ml[s].x);
    M = warp_max(M);
    float L = 0.f;
    for (int s = lane; s < ns; s += 32) if (ml[s].y > 0.f) L += exp2f(ml[s].x - M) * ml[s].y;
    L = warp_sum(L);
    const float inv = L > 0.f ? a.v_scale / L : 0.f;
    for (int s = lane; s < ns; s += 32) wsm[g * ns + s] = ml[s].y > 0.f ? exp2f(ml[s].x - M) * inv : 0.f;
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += kAttnThreads) {
    const int g = e / D, d = e - g * D;
    const float* po = a.part_o + (head0 + g) * ns * D + d;
    const float* wg = wsm + g * ns;
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    int s = 0;
    for (; s + 4 <= ns; s += 4) {
      const float w0 = wg[s], w1 = wg[s + 1], w2 = wg[s + 2], w3 = wg[s + 3];
      if (w0 != 0.f) acc0 += w0 * po[(size_t)s * D];
      if (w1 != 0.f) acc1 += w1 * po[(size_t)(s + 1) * D];
      if (w2 != 0.f) acc2 += w2 * po[(size_t)(s + 2) * D];
      if (w3 != 0.f) acc3 += w3 * po[(size_t)(s + 3) * D];
    }
    for (; s < ns; ++s) if (wg[s] != 0.f) acc0 += wg[s] * po[(size_t)s * D];
    const float o = (acc0 + acc1) + (acc2 + acc3);
    const size_t oi = (head0 + g) * D + d;
    if (a.out) a.out[oi] = o;
    if (a.out_hl) {                                // high/low BF16 rows for the tensor-core GEMM
      const size_t row = oi / ((size_t)a.nq * D), col = oi % ((size_t)a.nq * D);
      const bf16 h = __float2bfloat16_rn(o);
      a.out_hl[row * a.nq * D + col] = h;
      a.out_hl[(a.rp_hl + row) * a.nq * D + col] = __float2bfloat16_rn(o - __bfloat162float(h));
    }
  }
}

// Fused "RoPE + KV-cache write" ("Kernels, Fusion & CUDA Graphs", "Fix 1:
// kernel fusion"): rotate the new token's key for KV head h and store it and its
// value at block bt[p / 16], slot p % 16, rounded to the cache format.
template <int D, int KV8>
__device__ __forceinline__ void write_new_kv(const AttnArgs& a, int b, int h, int pos, int blk) {
  const int half = D / 2;
  const float* src = a.qkv + (size_t)b * a.ld_qkv;
  const int kcol = (a.nq + h) * D, vcol = (a.nq + a.nkv + h) * D;
  const float2* cs = a.rope + (size_t)pos * half;
  const size_t base = (((size_t)blk * a.nkv + h) * kBlockTokens + pos % kBlockTokens) * D;
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    float k1 = 0.f, k2 = 0.f, v = 0.f;
    const int ip = i < half ? i : i - half;
    for (int s2 = 0; s2 < a.qkv_nsplit; ++s2) {
      const float* p = src + (size_t)s2 * a.qkv_split_stride;
      k1 += p[kcol + ip];
      k2 += p[kcol + ip + half];
      v += p[vcol + i];
    }
    const float2 t = cs[ip];
    const float k = i < half ? k1 * t.x - k2 * t.y : k2 * t.x + k1 * t.y;
    const float ks = __fdiv_rn(k, a.k_scale), vs = __fdiv_rn(v, a.v_scale);
    if (KV8) {
      reinterpret_cast<uint8_t*>(const_cast<void*>(a.kpool))[base + i] = f32_to_e4m3(ks);
      reinterpret_cast<uint8_t*>(const_cast<void*>(a.vpool))[base + i] = f32_to_e4m3(vs);
    } else {
      reinterpret_cast<uint16_t*>(const_cast<void*>(a.kpool))[base + i] = f32_to_bf16_bits(ks);
      reinterpret_cast<uint16_t*>(const_cast<void*>(a.vpool))[base + i] = f32_to_bf16_bits(vs);
    }
  }
}

template <int D, int KV8>
__global__ void __launch_bounds__(kAttnThreads, 2) attn_split_kernel(const AttnArgs a) {
  using S = AttnShape<D, KV8>;
  extern __shared__ __align__(16) unsigned char smem[];
  const int sp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int G = a.nq / a.nkv;
  const int tid = threadIdx.x;
  const size_t head0 = (size_t)b * a.nq + (size_t)h * G;             // first query head of the group
  const int seq = a.seq_lens[b];
  pdl_launch_dependents();

  // The cached context is not produced by the previous kernel: pull this
  // split's K and V blocks into L2 before waiting for it.
  if (seq >= 1 && seq <= a.bt_stride * kBlockTokens) {
    const int nb_all = (seq + kBlockTokens - 1) / kBlockTokens;
    const int j = sp * a.bps + (tid >> 1);
    if ((tid >> 1) < a.bps && j < nb_all) {
      const int blk = a.bt[(size_t)b * a.bt_stride + j];
      if (blk >= 0 && blk <= a.num_blocks) {
        const size_t off = ((size_t)blk * a.nkv + h) * kBlockTokens * S::ROWB;
        prefetch_l2((const unsigned char*)((tid & 1) ? a.vpool : a.kpool) + off, kBlockTokens * S::ROWB);
      }
    }
  }
  pdl_wait();

  if (a.qkv) {
    // the split holding the new token's block writes its K and V first
    int pos = a.positions[b];
    const bool pos_ok = pos >= 0 && pos < a.max_pos;
    if (!pos_ok && tid == 0 && sp == 0 && h == 0) set_err(a.err, MBT_DEV_POS_RANGE);
    const int jb = pos_ok ? pos / kBlockTokens : -1;
    if (pos_ok && jb < a.bt_stride && sp == jb / a.bps) {
      const int blk = a.bt[(size_t)b * a.bt_stride + jb];
      if (blk >= 0 && blk <= a.num_blocks) write_new_kv<D, KV8>(a, b, h, pos, blk);
      else if (tid == 0) set_err(a.err, MBT_DEV_BLOCK_RANGE);
    } else if (pos_ok && jb >= a.bt_stride && tid == 0 && sp == 0) {
      set_err(a.err, MBT_DEV_BLOCK_RANGE);
    }
    __syncthreads();
  }
  const bool seq_ok = seq >= 1 && seq <= a.bt_stride * kBlockTokens;
  if (!seq_ok && tid == 0 && sp == 0 && h == 0) set_err(a.err, MBT_DEV_SEQLEN_RANGE);
  const int nblk = seq_ok ? (seq + kBlockTokens - 1) / kBlockTokens : 0;
  const int blk0 = sp * a.bps;
  const int blk1 = min(nblk, blk0 + a.bps);
  if (blk0 < nblk) attend<D, KV8>(a, smem, b, h, sp, G, head0, seq, blk0, blk1);
  else if (tid < G) a.part_ml[(head0 + tid) * a.nsplit + sp] = make_float2(-INFINITY, 0.f);

  // ticket: the last CTA of this (row, KV head) merges the splits
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int t = atomicAdd(a.tickets + (size_t)b * a.nkv + h, 1);
    last = (t == a.nsplit - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  merge_splits(a, reinterpret_cast<float*>(smem), G, head0, D);
  if (tid == 0) a.tickets[(size_t)b * a.nkv + h] = 0;     // ready for the next launch
}



void attn_plan(int B, int nkv, int max_blocks, int num_sms, int* bps, int* nsplit) {
  // Enough CTAs to cover the SMs, but at least two 64-token tiles per split so
  // that the double buffer overlaps loads with math and the merge stays short.
  const int target = num_sms;
  const int pairs = B * nkv;
  int want = (target + pairs - 1) / pairs;
  if (want < 1) want = 1;
  int per = (max_blocks + want - 1) / want;
  const int min_per = 2 * kAttnTile / kBlockTokens;
  if (per < min_per) per = min_per;
  if (per > max_blocks) per = max_blocks;
  if (per < 1) per = 1;
  *bps = per;
  *nsplit = (max_blocks + per - 1) / per;
}

namespace {
template <int D, int KV8>
void* attn_fn() { return (void*)attn_split_kernel<D, KV8>; }
void* attn_pick(int d, int kv8, size_t* smem) {
  if (d == 64) {
    *smem = kv8 ? AttnShape<64, 1>::SMEM : AttnShape<64, 0>::SMEM;
    return kv8 ? attn_fn<64, 1>() : attn_fn<64, 0>();
  }
  *smem = kv8 ? AttnShape<128, 1>::SMEM : AttnShape<128, 0>::SMEM;
  return kv8 ? attn_fn<128, 1>() : attn_fn<128, 0>();
}
}  // namespace

cudaError_t attn_init() {
  for (int d : {64, 128})
    for (int kv8 = 0; kv8 < 2; ++kv8) {
      size_t sm;
      void* fn = attn_pick(d, kv8, &sm);
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s) {
  size_t sm;
  void* fn = attn_pick(a.d, a.kv_fp8, &sm);
  AttnArgs args = a;
  void* params[] = {&args};
  return launch_pdl(fn, dim3(a.nsplit, a.nkv, a.B), dim3(kAttnThreads), sm, s, params);
}

}  // namespace mbt
