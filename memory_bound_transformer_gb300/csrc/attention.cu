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
constexpr int kMaxSplitBlocks = 512;   // KV blocks one split may cover (8192 tokens)

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
  static constexpr int ROWB = D * ESZ;               // bytes of one token's K (or V) for one head in the cache
  static constexpr int NCH = ROWB / 16;              // 16-byte chunks per cache row
  static constexpr int BROWB = D * 2;                // bytes per token row of a BF16 compute tile
  static constexpr int BNCH = BROWB / 16;            // 16-byte chunks per BF16 row (8 or 16)
  static constexpr int KSTEPS = D / 16;              // MMA k-steps over d for Q K^T
  static constexpr int DT = D / 8;                   // 8-wide d tiles of the output
  static constexpr size_t Q_BYTES = (size_t)16 * D * 4;
  static constexpr size_t T_BYTES = (size_t)kAttnTile * BROWB;
  static constexpr size_t R_BYTES = (size_t)kAttnTile * ROWB;
  static constexpr size_t SMEM = Q_BYTES + 4 * T_BYTES + (KV8 ? 4 * R_BYTES : 0);
};

// 16 e4m3 codes -> 16 floats, exactly.
template <int KV8>
__device__ __forceinline__ void chunk_to_float(const uint4& c, float* f);
template <>
__device__ __forceinline__ void chunk_to_float<1>(const uint4& c, float* f) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 a = e4m3x2_to_float2(w[i]), b = e4m3x2_to_float2(w[i] >> 16);
    f[4 * i] = a.x; f[4 * i + 1] = a.y; f[4 * i + 2] = b.x; f[4 * i + 3] = b.y;
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return a | (b << 16);
}
// x = hi + lo: the BF16 high part and the BF16 rounding of the remainder.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const bf16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  hi = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
  lo = pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
// D += A (16x16 BF16, row) * B (16x8 BF16, col), fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One split of one (row, KV head): stream its KV blocks once for all query
// heads of the group and leave (unnormalised o, running max m, sum l) per head.
// The group's query heads are the 16 rows of the MMA tiles (padded with zero
// rows); each warp takes 16 tokens of every 64-token tile: S = Q K^T and
// O += P V on the tensor cores with Q and P split into BF16 high + low parts
// (fp32-level accuracy), the online softmax in registers, and the four warps'
// states merged at the end.
template <int D, int KV8>
__device__ __forceinline__ void attend(const AttnArgs& a, unsigned char* smem, int b, int h, int sp,
                                       int G, size_t head0, int seq, int blk0, int blk1) {
  using S = AttnShape<D, KV8>;
  float* qs = reinterpret_cast<float*>(smem);                        // [16][D], rows >= G are zero
  unsigned char* kbf = smem + S::Q_BYTES;                             // [2][tile][BROWB] BF16, swizzled
  unsigned char* vbf = kbf + 2 * S::T_BYTES;
  unsigned char* raw = vbf + 2 * S::T_BYTES;                          // e4m3 caches: [2][K|V][tile][ROWB]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;

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
      const int gg = e / half, i = e - gg * half;
      float x1 = 0.f, x2 = 0.f;
      for (int s2 = 0; s2 < a.qkv_nsplit; ++s2) {
        x1 += src[(size_t)s2 * a.qkv_split_stride + gg * D + i];
        x2 += src[(size_t)s2 * a.qkv_split_stride + gg * D + i + half];
      }
      const float2 t = cs[i];
      qs[gg * D + i] = (x1 * t.x - x2 * t.y) * qscale;
      qs[gg * D + i + half] = (x2 * t.x + x1 * t.y) * qscale;
    }
  } else {
    for (int i = tid; i < G * D; i += kAttnThreads) qs[i] = a.q[head0 * D + i] * qscale;
  }
  for (int i = G * D + tid; i < 16 * D; i += kAttnThreads) qs[i] = 0.f;

  const unsigned char* kpool = reinterpret_cast<const unsigned char*>(a.kpool);
  const unsigned char* vpool = reinterpret_cast<const unsigned char*>(a.vpool);
  // this split's block ids, staged once in shared memory (validated here)
  __shared__ int sblk[kMaxSplitBlocks];
  const int* bt = a.bt + (size_t)b * a.bt_stride;
  for (int j = tid; j < blk1 - blk0; j += kAttnThreads) {
    int blk = bt[blk0 + j];
    if (blk < 0 || blk > a.num_blocks) {
      set_err(a.err, MBT_DEV_BLOCK_RANGE);
      blk = a.num_blocks;
    }
    sblk[j] = blk;
  }
  const int tok_begin = blk0 * kBlockTokens;
  const int tok_end_blk = blk1 * kBlockTokens;                       // whole blocks loaded
  const int ntiles = (tok_end_blk - tok_begin + kAttnTile - 1) / kAttnTile;

  auto load_tile = [&](int t, int buf) {
    const int tok0 = tok_begin + t * kAttnTile;
    const int rows = min(kAttnTile, tok_end_blk - tok0);
    unsigned char* kd = KV8 ? raw + (size_t)buf * 2 * S::R_BYTES : kbf + (size_t)buf * S::T_BYTES;
    unsigned char* vd = KV8 ? kd + S::R_BYTES : vbf + (size_t)buf * S::T_BYTES;
    for (int i = tid; i < rows * S::NCH; i += kAttnThreads) {
      const int row = i / S::NCH, ch = i - row * S::NCH;
      const int tok = tok0 + row;
      const int blk = sblk[tok / kBlockTokens - blk0];
      const size_t off = (((size_t)blk * a.nkv + h) * kBlockTokens + (tok % kBlockTokens)) * S::ROWB + ch * 16;
      const int sch = KV8 ? ch : (ch ^ (row & 7));                   // BF16 tiles are swizzled in place
      cp_async16(kd + row * S::ROWB + sch * 16, kpool + off);
      cp_async16(vd + row * S::ROWB + sch * 16, vpool + off);
    }
    cp_async_commit();
  };

  __syncthreads();                                                    // qs and block ids complete
  load_tile(0, 0);

  // Q fragments (A operand, rows = query heads, k = d), high and low parts
  uint32_t qh[S::KSTEPS][4], ql[S::KSTEPS][4];
#pragma unroll
  for (int kk = 0; kk < S::KSTEPS; ++kk)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = g + (r & 1) * 8, col = 16 * kk + 2 * t4 + (r >> 1) * 8;
      split_bf16(qs[row * D + col], qs[row * D + col + 1], qh[kk][r], ql[kk][r]);
    }

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;          // rows g and g + 8
  float o[S::DT][4];
#pragma unroll
  for (int i = 0; i < S::DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1;
    if (t + 1 < ntiles) { load_tile(t + 1, buf ^ 1); cp_async_wait<1>(); }
    else cp_async_wait<0>();
    __syncthreads();
    const int tok0 = tok_begin + t * kAttnTile;
    const int nvalid = min(kAttnTile, min(seq, tok_end_blk) - tok0);   // this split's tokens only
    unsigned char* kt = kbf + (size_t)buf * S::T_BYTES;
    unsigned char* vt = vbf + (size_t)buf * S::T_BYTES;
    if (KV8) {
      // widen the e4m3 tile to BF16 (exact), swizzled; rows past the context are zero
      const unsigned char* rk = raw + (size_t)buf * 2 * S::R_BYTES;
      for (int i = tid; i < 2 * kAttnTile * S::NCH; i += kAttnThreads) {
        const int which = i / (kAttnTile * S::NCH), j = i - which * kAttnTile * S::NCH;
        const int row = j / S::NCH, ch = j - row * S::NCH;
        uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
        if (row < nvalid) {
          const uint4 c = *reinterpret_cast<const uint4*>(rk + which * S::R_BYTES + row * S::ROWB + ch * 16);
          float f[16];
          chunk_to_float<1>(c, f);
          lo = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
          hi = make_uint4(pack_bf16(f[8], f[9]), pack_bf16(f[10], f[11]), pack_bf16(f[12], f[13]), pack_bf16(f[14], f[15]));
        }
        unsigned char* dst = (which ? vt : kt) + row * S::BROWB;
        *reinterpret_cast<uint4*>(dst + (((2 * ch) ^ (row & 7)) * 16)) = lo;
        *reinterpret_cast<uint4*>(dst + (((2 * ch + 1) ^ (row & 7)) * 16)) = hi;
      }
      __syncthreads();
    } else if (nvalid < kAttnTile) {
      // rows past the context hold whatever the pool had: zero V so that P = 0 stays 0
      for (int i = tid; i < (kAttnTile - nvalid) * S::BNCH; i += kAttnThreads) {
        const int row = nvalid + i / S::BNCH, ch = i % S::BNCH;
        *reinterpret_cast<uint4*>(vt + row * S::BROWB + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
    }

    const int n0 = 16 * warp;                                         // this warp's tokens in the tile
    if (n0 < nvalid) {
      const uint32_t kbase = (uint32_t)__cvta_generic_to_shared(kt);
      const uint32_t vbase = (uint32_t)__cvta_generic_to_shared(vt);
      const int lm = lane >> 3, lr = lane & 7;
      // S = Q K^T over 16 tokens (two 8-token n-tiles)
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int krow = n0 + (lm >> 1) * 8 + lr;
#pragma unroll
        for (int kk = 0; kk < S::KSTEPS; ++kk) {
          uint32_t kf[4];
          const int ch = 2 * kk + (lm & 1);
          ldsm_x4(kbase + krow * S::BROWB + ((ch ^ (krow & 7)) * 16), kf);
          mma16816(sacc[0], qh[kk], kf[0], kf[1]);
          mma16816(sacc[0], ql[kk], kf[0], kf[1]);
          mma16816(sacc[1], qh[kk], kf[2], kf[3]);
          mma16816(sacc[1], ql[kk], kf[2], kf[3]);
        }
      }
      // mask, online softmax per query-head row (quad of lanes holds a row)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int tok = n0 + 8 * j + 2 * t4 + (c & 1);
          if (tok >= nvalid) sacc[j][c] = -INFINITY;
          if (c < 2) mx0 = fmaxf(mx0, sacc[j][c]); else mx1 = fmaxf(mx1, sacc[j][c]);
        }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float p = exp2f(sacc[j][c] - (c < 2 ? mu0 : mu1));
          sacc[j][c] = p;
          if (c < 2) ps0 += p; else ps1 += p;
        }
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
      l0 = l0 * al0 + ps0;
      l1 = l1 * al1 + ps1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int i = 0; i < S::DT; ++i) { o[i][0] *= al0; o[i][1] *= al0; o[i][2] *= al1; o[i][3] *= al1; }
      // P as the A operand (rows = heads, k = the 16 tokens), high and low parts
      uint32_t ph[4], pl[4];
      split_bf16(sacc[0][0], sacc[0][1], ph[0], pl[0]);
      split_bf16(sacc[0][2], sacc[0][3], ph[1], pl[1]);
      split_bf16(sacc[1][0], sacc[1][1], ph[2], pl[2]);
      split_bf16(sacc[1][2], sacc[1][3], ph[3], pl[3]);
      // O += P V (V fragments transposed out of the swizzled tile)
      const int vrow = n0 + (lm & 1) * 8 + lr;
#pragma unroll
      for (int dp = 0; dp < S::DT / 2; ++dp) {
        uint32_t vf[4];
        const int ch = 2 * dp + (lm >> 1);
        ldsm_x4_t(vbase + vrow * S::BROWB + ((ch ^ (vrow & 7)) * 16), vf);
        mma16816(o[2 * dp], ph, vf[0], vf[1]);
        mma16816(o[2 * dp], pl, vf[0], vf[1]);
        mma16816(o[2 * dp + 1], ph, vf[2], vf[3]);
        mma16816(o[2 * dp + 1], pl, vf[2], vf[3]);
      }
    }
    __syncthreads();
  }

  // merge the four warps' (m, l, o) per head row and write this split's partial
  float* sm_m = reinterpret_cast<float*>(kbf);                        // [4][16]
  float* sm_l = sm_m + 4 * 16;
  float* sm_o = sm_l + 4 * 16;                                        // [4][16][D]
  if (t4 == 0) {
    sm_m[warp * 16 + g] = m0; sm_m[warp * 16 + g + 8] = m1;
    sm_l[warp * 16 + g] = l0; sm_l[warp * 16 + g + 8] = l1;
  }
#pragma unroll
  for (int i = 0; i < S::DT; ++i) {
    const int d0 = 8 * i + 2 * t4;
    sm_o[(warp * 16 + g) * D + d0] = o[i][0];
    sm_o[(warp * 16 + g) * D + d0 + 1] = o[i][1];
    sm_o[(warp * 16 + g + 8) * D + d0] = o[i][2];
    sm_o[(warp * 16 + g + 8) * D + d0 + 1] = o[i][3];
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += kAttnThreads) {
    const int hr = e / D, d = e - hr * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) if (sm_l[w * 16 + hr] > 0.f) M = fmaxf(M, sm_m[w * 16 + hr]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (sm_l[w * 16 + hr] > 0.f) {
        const float sc = exp2f(sm_m[w * 16 + hr] - M);
        L += sm_l[w * 16 + hr] * sc;
        acc += sm_o[(w * 16 + hr) * D + d] * sc;
      }
    }
    a.part_o[((head0 + hr) * a.nsplit + sp) * D + d] = acc;
    if (d == 0) a.part_ml[(head0 + hr) * a.nsplit + sp] = make_float2(L > 0.f ? M : -INFINITY, L);
  }
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
    // only the first two tiles: at large batches all CTAs' splits together
    // exceed L2 and a deeper prefetch would be evicted before use
    const int pf = min(a.bps, 2 * kAttnTile / kBlockTokens);
    if ((tid >> 1) < pf && j < nb_all) {
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
  // About four CTAs per SM so that rows with long contexts do not form the
  // tail (contexts in one batch differ by up to 8x), but at least two 64-token
  // tiles per split so that the double buffer overlaps loads with math and
  // the merge stays short.
  const int target = 4 * num_sms;
  const int pairs = B * nkv;
  int want = (target + pairs - 1) / pairs;
  if (want < 1) want = 1;
  int per = (max_blocks + want - 1) / want;
  const int min_per = 2 * kAttnTile / kBlockTokens;
  if (per < min_per) per = min_per;
  if (per > max_blocks) per = max_blocks;
  if (per > kMaxSplitBlocks) per = kMaxSplitBlocks;
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
