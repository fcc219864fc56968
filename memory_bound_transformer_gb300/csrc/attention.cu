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
// running max and sum per head and writes an unnormalised partial. With four
// to eight splits the splits of a (row, KV head) are one thread-block cluster
// and the first of them merges the others' partials through distributed
// shared memory after a cluster barrier; otherwise the last CTA of the group to
// finish -- found with an atomic ticket, nothing waits -- merges them from
// global memory.
#include "common.cuh"
#include "internal.h"

namespace mbt {

// Fewest 64-token tiles per context split.
#ifndef MBT_ATTN_MIN_TILES
#define MBT_ATTN_MIN_TILES 2
#endif
constexpr int kAttnThreads = 128;
constexpr int kAttnTile = 64;      // tokens per shared-memory tile (4 blocks)
constexpr int kMaxSplitBlocks = 512;   // KV blocks one split may cover (8192 tokens)
constexpr int kAttnCluster = 8;        // most splits per (row, KV head): a portable cluster

__device__ __forceinline__ void cp_async16(void* s, const void* g) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(s);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

template <int D, int KV8, int NT = 1, int O4 = 0>
struct AttnShape {
  static constexpr int ESZ = KV8 ? 1 : 2;
  static constexpr int ROWB = D * ESZ;               // bytes of one token's K (or V) for one head in the cache
  static constexpr int NCH = ROWB / 16;              // 16-byte chunks per cache row
  static constexpr int BROWB = D * 2;                // bytes per token row of a BF16 compute tile
  static constexpr int BNCH = BROWB / 16;            // 16-byte chunks per BF16 row (8 or 16)
  static constexpr int KSTEPS = D / 16;              // MMA k-steps over d for Q K^T
  static constexpr int MT = D / 16;                  // 16-row d tiles of O^T
  static constexpr size_t T_BYTES = (size_t)kAttnTile * BROWB;
  static constexpr size_t R_BYTES = (size_t)kAttnTile * ROWB;
  // BF16 caches: K and V tiles double-buffered in place. e4m3 caches: raw
  // (K, V) tiles in flight (half the bytes of a BF16 tile); K is widened into
  // MMA fragments straight from its raw tile, V into one FP16 tile. The O4
  // form of the e4m3 kernel with up to 8 query heads (one n-tile) fits four
  // CTAs per SM (two raw stages, 8 query rows, <= 128 registers), which lets
  // batch 64 x 8 KV heads run as one wave of single-split CTAs; small grids
  // (batch 1-4) keep three stages, three CTAs per SM, whose deeper prologue
  // (three tiles requested before the PDL wait) their latency wants.
  static constexpr bool OCC4 = O4 && KV8 && NT == 1;
  static constexpr int MINB = OCC4 ? 4 : 3;
  static constexpr int QROWS = OCC4 ? 8 : 16;         // query rows of the tile (G <= QROWS)
  static constexpr size_t Q_BYTES = (size_t)QROWS * D * 4;
  static constexpr int NBUF = KV8 ? 0 : 2;
  static constexpr int NRAW = KV8 ? (OCC4 ? 2 : 3) : 0;
  static constexpr int NPRO = KV8 ? NRAW : 2;          // tiles requested before the PDL wait
  static constexpr size_t SMEM = Q_BYTES + (KV8 ? T_BYTES : 2 * NBUF * T_BYTES) + (size_t)NRAW * 2 * R_BYTES;
};

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
// Transpose of an 8x8 16-bit matrix held one row pair per lane (mma fragment layout).
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// x = hi + lo in FP16 (used with e4m3 caches, whose codes widen to FP16 exactly)
__device__ __forceinline__ void split_f16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
  hi = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
  const __half l0 = __float2half_rn(x0 - __half2float(h0)), l1 = __float2half_rn(x1 - __half2float(h1));
  lo = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
}
template <int F16>
__device__ __forceinline__ void split_hl(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  if (F16) split_f16(x0, x1, hi, lo);
  else split_bf16(x0, x1, hi, lo);
}

// D += A (16x16, row) * B (16x8, col), fp32 accumulate; BF16 or FP16 operands.
template <int F16>
__device__ __forceinline__ void mma_t(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if (F16)
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Loads two floats from the shared memory of CTA `rank` of the cluster, at the
// address that p has in this CTA.
__device__ __forceinline__ float2 ld_dsmem_f2(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(r) : "memory");
  return v;
}

// Fused "RoPE + KV-cache write" ("Kernels, Fusion & CUDA Graphs", "Fix 1:
// kernel fusion"): rotate the new token's key for KV head h and store it and its
// value at block bt[p / 16], slot p % 16, rounded to the cache format. Thread
// i < D handles element i and returns its two codes (for a copy in shared memory).
template <int D, int KV8>
__device__ __forceinline__ void write_new_kv(const AttnArgs& a, int b, int h, int pos, int blk,
                                             uint32_t& kcode, uint32_t& vcode) {
  static_assert(D <= kAttnThreads, "one element per thread");
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
      kcode = f32_to_e4m3(ks);
      vcode = f32_to_e4m3(vs);
      reinterpret_cast<uint8_t*>(const_cast<void*>(a.kpool))[base + i] = (uint8_t)kcode;
      reinterpret_cast<uint8_t*>(const_cast<void*>(a.vpool))[base + i] = (uint8_t)vcode;
    } else {
      kcode = f32_to_bf16_bits(ks);
      vcode = f32_to_bf16_bits(vs);
      reinterpret_cast<uint16_t*>(const_cast<void*>(a.kpool))[base + i] = (uint16_t)kcode;
      reinterpret_cast<uint16_t*>(const_cast<void*>(a.vpool))[base + i] = (uint16_t)vcode;
    }
  }
}

// One split of one (row, KV head): stream its KV blocks once for all query
// heads of the group and leave (unnormalised o, running max m, sum l) per head.
// Each warp takes 16 tokens of every 64-token tile; the group's query heads
// are the N dimension of the MMA tiles (8 per n-tile, zero-padded):
// S^T = K Q^T and O^T += V^T P^T on the tensor cores with Q and P split into
// BF16 high + low parts (fp32-level accuracy), the online softmax in
// registers, and the four warps' states merged at the end.
//
// The cached context does not depend on the previous kernel (only this
// kernel writes this layer's cache, and a step starts after the previous one
// has finished), so the block ids and the first two tiles are requested
// before the wait on the QKV projection. The new token's row, which this CTA
// writes after the wait, is patched into a tile already in shared memory
// (tiles loaded later read it from the cache).
// One element of the attention output (index oi of [B][nq * D]): fp32, and/or
// the 16-bit high/low rows the next tensor-core projection reads.
__device__ __forceinline__ void store_attn_out(const AttnArgs& a, size_t oi, int D, float o) {
  if (a.out) a.out[oi] = o;
  if (a.out_hl) {
    const size_t row = oi / ((size_t)a.nq * D), col = oi % ((size_t)a.nq * D);
    uint16_t* hl = reinterpret_cast<uint16_t*>(a.out_hl);
    const float hv = a.hl_f16 ? __half2float(__float2half_rn(o)) : __bfloat162float(__float2bfloat16_rn(o));
    hl[row * a.nq * D + col] = a.hl_f16 ? __half_as_ushort(__float2half_rn(o))
                                        : __bfloat16_as_ushort(__float2bfloat16_rn(o));
    hl[(a.rp_hl + row) * a.nq * D + col] = a.hl_f16 ? __half_as_ushort(__float2half_rn(o - hv))
                                                     : __bfloat16_as_ushort(__float2bfloat16_rn(o - hv));
  }
}

template <int D, int KV8, int NT, int CL, int O4>
__device__ __forceinline__ void attend(const AttnArgs& a, unsigned char* smem, int b, int h, int sp,
                                       int G, size_t head0, int seq, int blk0, int blk1, bool writer,
                                       int pos, int wblk, float2* cl_ml) {
  using S = AttnShape<D, KV8, NT, O4>;
  float* qs = reinterpret_cast<float*>(smem);                        // [16][D], rows >= G are zero
  unsigned char* kbf = smem + S::Q_BYTES;                             // BF16: [NBUF][tile][BROWB], swizzled
  unsigned char* vbf = KV8 ? kbf : kbf + S::NBUF * S::T_BYTES;        // BF16: V tiles; e4m3: the FP16 V tile
  unsigned char* raw = vbf + (KV8 ? S::T_BYTES : S::NBUF * S::T_BYTES);   // e4m3: [NRAW][K|V][tile][ROWB]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;

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
  // tile of this split that holds the new token (written below), else -1
  const int tnew = (writer && pos >= tok_begin && pos < tok_end_blk) ? (pos - tok_begin) / kAttnTile : -1;

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
      // BF16 tiles are swizzled in place; the raw e4m3 K tile too (its
      // fragments are read straight from it), the raw V tile is not
      const int ksch = KV8 ? (ch ^ (row & (S::NCH - 1))) : (ch ^ (row & 7));
      const int vsch = KV8 ? ch : (ch ^ (row & 7));
      cp_async16(kd + row * S::ROWB + ksch * 16, kpool + off);
      cp_async16(vd + row * S::ROWB + vsch * 16, vpool + off);
    }
    cp_async_commit();
  };

  __syncthreads();                                                    // block ids complete
  for (int t = 0; t < S::NPRO && t < ntiles; ++t) load_tile(t, t);
  // the next two tiles towards L2
  if (ntiles > S::NPRO) {
    const int j = S::NPRO * kAttnTile / kBlockTokens + (tid >> 1);
    if ((tid >> 1) < 2 * kAttnTile / kBlockTokens && j < blk1 - blk0) {
      const size_t off = ((size_t)sblk[j] * a.nkv + h) * kBlockTokens * S::ROWB;
      prefetch_l2((const unsigned char*)((tid & 1) ? a.vpool : a.kpool) + off, kBlockTokens * S::ROWB);
    }
  }

  // the query rotation's cos/sin at this row's position: a step input and a
  // table, neither written by the previous kernel, so loaded before the wait
  constexpr int QE = 16 * (D / 2) / kAttnThreads;                     // elements per thread at G <= 16
  float2 tc[QE];
  if (a.qkv) {
    const int half = D / 2;
    int qpos = a.positions[b];
    if (qpos < 0 || qpos >= a.max_pos) qpos = 0;
    const float2* cs = a.rope + (size_t)qpos * half;
#pragma unroll
    for (int j = 0; j < QE; ++j) {
      const int e = tid + j * kAttnThreads;
      tc[j] = e < G * half ? cs[e % half] : make_float2(0.f, 0.f);
    }
  }

  pdl_wait();

  if (writer) {
    // the new token's K (rotated) and V go into the cache, and into the tile
    // already requested when it is one of those requested before the wait
    uint32_t kc = 0, vc = 0;
    write_new_kv<D, KV8>(a, b, h, pos, wblk, kc, vc);
    if (tnew >= 0 && tnew < S::NPRO) {
      cp_async_wait<0>();
      __syncthreads();                                                // the tile's copies have landed
      const int r = pos - (tok_begin + tnew * kAttnTile);
      if (tid < D) {
        if (KV8) {
          unsigned char* rk = raw + (size_t)tnew * 2 * S::R_BYTES + (size_t)r * S::ROWB;
          rk[(((tid >> 4) ^ (r & (S::NCH - 1))) << 4) + (tid & 15)] = (unsigned char)kc;
          rk[S::R_BYTES + tid] = (unsigned char)vc;
        } else {
          const size_t off = (size_t)tnew * S::T_BYTES + (size_t)r * S::BROWB +
                             (size_t)(((tid >> 3) ^ (r & 7)) * 16 + (tid & 7) * 2);
          *reinterpret_cast<uint16_t*>(kbf + off) = (uint16_t)kc;
          *reinterpret_cast<uint16_t*>(vbf + off) = (uint16_t)vc;
        }
      }
    }
  }

  // queries of the group, pre-scaled into the log2 domain with the K dequant scale
  // (e4m3 caches: Q is split in FP16, so the K scale is applied to the fp32
  // scores instead, keeping Q's range independent of it)
  const float qscale = 1.4426950408889634f / sqrtf((float)D) * (KV8 ? 1.f : a.k_scale);
  const float sscale = KV8 ? a.k_scale : 1.f;
  if (a.qkv) {
    // RoPE (rotate-half: element i pairs with i + D/2) straight from the QKV
    // projection's partial sums
    const int half = D / 2;
    const float* src = a.qkv + (size_t)b * a.ld_qkv + (size_t)h * G * D;
    // every load of the thread's elements first (one round trip), then the rotation
    float x1[QE], x2[QE];
#pragma unroll
    for (int j = 0; j < QE; ++j) {
      const int e = tid + j * kAttnThreads;
      x1[j] = 0.f; x2[j] = 0.f;
      if (e < G * half) {
        const int gg = e / half, i = e - gg * half;
        for (int s2 = 0; s2 < a.qkv_nsplit; ++s2) {
          x1[j] += src[(size_t)s2 * a.qkv_split_stride + gg * D + i];
          x2[j] += src[(size_t)s2 * a.qkv_split_stride + gg * D + i + half];
        }
      }
    }
#pragma unroll
    for (int j = 0; j < QE; ++j) {
      const int e = tid + j * kAttnThreads;
      if (e < G * half) {
        const int gg = e / half, i = e - gg * half;
        qs[gg * D + i] = (x1[j] * tc[j].x - x2[j] * tc[j].y) * qscale;
        qs[gg * D + i + half] = (x2[j] * tc[j].x + x1[j] * tc[j].y) * qscale;
      }
    }
  } else {
    for (int i = tid; i < G * D; i += kAttnThreads) qs[i] = a.q[head0 * D + i] * qscale;
  }
  for (int i = G * D + tid; i < S::QROWS * D; i += kAttnThreads) qs[i] = 0.f;
  __syncthreads();                                                    // qs complete

  // Q^T fragments (B operand: k = d, n = query head), high and low parts, in
  // NT n-tiles of 8 heads (heads >= G are the zero rows of qs)
  uint32_t qh[NT][S::KSTEPS][2], ql[NT][S::KSTEPS][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int kk = 0; kk < S::KSTEPS; ++kk)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int head = nt * 8 + g, col = 16 * kk + 2 * t4 + r * 8;
        split_hl<KV8>(qs[head * D + col], qs[head * D + col + 1], qh[nt][kk][r], ql[nt][kk][r]);
      }

  // softmax state of this thread's two heads per n-tile (nt*8 + 2*t4, +1),
  // the same in every lane of a column group
  float mst[NT][2], lst[NT][2];
  float o[NT][S::MT][4];                                              // O^T: 16 d x 8 heads per m-tile
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    mst[nt][0] = mst[nt][1] = -INFINITY;
    lst[nt][0] = lst[nt][1] = 0.f;
#pragma unroll
    for (int i = 0; i < S::MT; ++i) o[nt][i][0] = o[nt][i][1] = o[nt][i][2] = o[nt][i][3] = 0.f;
  }

  constexpr int NR = S::NRAW > 0 ? S::NRAW : 1;
  for (int t = 0; t < ntiles; ++t) {
    const int buf = KV8 ? t % NR : (t & 1);
    if (KV8) {
      // tiles 0 .. NRAW-1 were requested up front; from tile 1 on, tile
      // t + NRAW - 1 goes into the stage tile t - 1 has left
      if (t >= 1 && t + NR - 1 < ntiles) load_tile(t + NR - 1, (t + NR - 1) % NR);
      const int after = min(NR - 1, ntiles - 1 - t);                   // copy groups still allowed in flight
      if (after >= 2) cp_async_wait<2>();
      else if (after == 1) cp_async_wait<1>();
      else cp_async_wait<0>();
    } else {
      // tiles 0 and 1 were requested up front; from tile 1 on, the tile after
      // next goes into the buffer the previous tile has left
      if (t >= 1 && t + 1 < ntiles) { load_tile(t + 1, buf ^ 1); cp_async_wait<1>(); }
      else cp_async_wait<0>();
    }
    __syncthreads();
    const int tok0 = tok_begin + t * kAttnTile;
    const int nvalid = min(kAttnTile, min(seq, tok_end_blk) - tok0);   // this split's tokens only
    unsigned char* kt = kbf + (size_t)(KV8 ? 0 : buf) * S::T_BYTES;
    unsigned char* vt = vbf + (size_t)(KV8 ? 0 : buf) * S::T_BYTES;
    const unsigned char* rk = raw + (size_t)buf * 2 * S::R_BYTES;      // e4m3: this tile's raw K, then V
    if (KV8) {
      // widen the e4m3 V tile to FP16 (exact, one conversion per two codes),
      // swizzled; rows past the context are zero
      for (int i = tid; i < kAttnTile * S::NCH; i += kAttnThreads) {
        const int row = i / S::NCH, ch = i - row * S::NCH;
        uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
        if (row < nvalid) {
          const uint4 c = *reinterpret_cast<const uint4*>(rk + S::R_BYTES + row * S::ROWB + ch * 16);
          lo = make_uint4(e4m3x2_to_h2bits(c.x), e4m3x2_to_h2bits(c.x >> 16), e4m3x2_to_h2bits(c.y),
                          e4m3x2_to_h2bits(c.y >> 16));
          hi = make_uint4(e4m3x2_to_h2bits(c.z), e4m3x2_to_h2bits(c.z >> 16), e4m3x2_to_h2bits(c.w),
                          e4m3x2_to_h2bits(c.w >> 16));
        }
        unsigned char* dst = vt + row * S::BROWB;
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
      // S^T [16 tokens x 8 heads] = K Q^T: K rows are the A operand
      float st[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) st[nt][0] = st[nt][1] = st[nt][2] = st[nt][3] = 0.f;
      {
        const int krow = n0 + (lm & 1) * 8 + lr;
#pragma unroll
        for (int kk = 0; kk < S::KSTEPS; ++kk) {
          uint32_t kf[4];
          if (KV8) {
            // the A fragment (rows g, g + 8; columns 2 t4, 2 t4 + 8 of this
            // 16-wide k step) widened from the raw, swizzled K tile
            const int ra = n0 + g, rb = ra + 8, c0 = 16 * kk + 2 * t4;
            auto code2 = [&](int r, int c) {
              return (uint32_t)*reinterpret_cast<const uint16_t*>(
                  rk + r * S::ROWB + ((((c >> 4) ^ (r & (S::NCH - 1)))) << 4) + (c & 15));
            };
            kf[0] = e4m3x2_to_h2bits(code2(ra, c0));
            kf[1] = e4m3x2_to_h2bits(code2(rb, c0));
            kf[2] = e4m3x2_to_h2bits(code2(ra, c0 + 8));
            kf[3] = e4m3x2_to_h2bits(code2(rb, c0 + 8));
          } else {
            const int ch = 2 * kk + (lm >> 1);
            ldsm_x4(kbase + krow * S::BROWB + ((ch ^ (krow & 7)) * 16), kf);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_t<KV8>(st[nt], kf, qh[nt][kk][0], qh[nt][kk][1]);
            mma_t<KV8>(st[nt], kf, ql[nt][kk][0], ql[nt][kk][1]);
          }
        }
      }
      const bool v0 = n0 + g < nvalid, v1 = n0 + g + 8 < nvalid;     // tokens of c0/c1 and c2/c3
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (KV8) { st[nt][0] *= sscale; st[nt][1] *= sscale; st[nt][2] *= sscale; st[nt][3] *= sscale; }
        if (!v0) { st[nt][0] = -INFINITY; st[nt][1] = -INFINITY; }
        if (!v1) { st[nt][2] = -INFINITY; st[nt][3] = -INFINITY; }
        // online softmax per head: the 16 tokens of a column sit in the 8 lanes of one t4
        float mx[2] = {fmaxf(st[nt][0], st[nt][2]), fmaxf(st[nt][1], st[nt][3])};
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], off));
        float al[2], ps[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const float mn = fmaxf(mst[nt][c], mx[c]);
          const float mu = mn == -INFINITY ? 0.f : mn;
          al[c] = exp2f(mst[nt][c] - mu);
          const float pa = exp2f(st[nt][c] - mu), pb = exp2f(st[nt][c + 2] - mu);
          st[nt][c] = pa;
          st[nt][c + 2] = pb;
          ps[c] = pa + pb;
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) ps[c] += __shfl_xor_sync(0xffffffffu, ps[c], off);
          lst[nt][c] = lst[nt][c] * al[c] + ps[c];
          mst[nt][c] = mn;
        }
#pragma unroll
        for (int i = 0; i < S::MT; ++i) {
          o[nt][i][0] *= al[0]; o[nt][i][1] *= al[1]; o[nt][i][2] *= al[0]; o[nt][i][3] *= al[1];
        }
      }
      // P^T as the B operand (k = tokens, n = heads): transpose the 8x8 BF16
      // halves of the S^T accumulator in registers; high and low parts
      uint32_t ph[NT][2], pl[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        uint32_t h0, l0, h1, l1;
        split_hl<KV8>(st[nt][0], st[nt][1], h0, l0);
        split_hl<KV8>(st[nt][2], st[nt][3], h1, l1);
        ph[nt][0] = movm_t(h0); ph[nt][1] = movm_t(h1);
        pl[nt][0] = movm_t(l0); pl[nt][1] = movm_t(l1);
      }
      // O^T [16 d x 8 heads] += V^T P^T: V^T fragments read transposed from the tile
      const int vrow = n0 + (lm >> 1) * 8 + lr;
#pragma unroll
      for (int mt = 0; mt < S::MT; ++mt) {
        uint32_t vf[4];
        const int ch = 2 * mt + (lm & 1);
        ldsm_x4_t(vbase + vrow * S::BROWB + ((ch ^ (vrow & 7)) * 16), vf);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_t<KV8>(o[nt][mt], vf, ph[nt][0], ph[nt][1]);
          mma_t<KV8>(o[nt][mt], vf, pl[nt][0], pl[nt][1]);
        }
      }
    }
    __syncthreads();
  }

  // merge the four warps' (m, l, o) per head and write this split's partial
  float* sm_m = reinterpret_cast<float*>(smem + S::Q_BYTES);          // [4][16]
  float* sm_l = sm_m + 4 * 16;
  float* sm_o = sm_l + 4 * 16;                                        // [4][16][D]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h0 = nt * 8 + 2 * t4;
    if (g == 0) {
      sm_m[warp * 16 + h0] = mst[nt][0]; sm_m[warp * 16 + h0 + 1] = mst[nt][1];
      sm_l[warp * 16 + h0] = lst[nt][0]; sm_l[warp * 16 + h0 + 1] = lst[nt][1];
    }
#pragma unroll
    for (int i = 0; i < S::MT; ++i) {
      const int d0 = 16 * i + g;
      sm_o[(warp * 16 + h0) * D + d0] = o[nt][i][0];
      sm_o[(warp * 16 + h0 + 1) * D + d0] = o[nt][i][1];
      sm_o[(warp * 16 + h0) * D + d0 + 8] = o[nt][i][2];
      sm_o[(warp * 16 + h0 + 1) * D + d0 + 8] = o[nt][i][3];
    }
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
    if (CL) {
      // the cluster's merging CTA reads it from this CTA's shared memory (the
      // query tile, no longer needed)
      qs[hr * D + d] = acc;
      if (d == 0) cl_ml[hr] = make_float2(L > 0.f ? M : -INFINITY, L);
    } else if (a.nsplit == 1) {
      // one split: the output itself (the same arithmetic as the merge of one)
      store_attn_out(a, (head0 + hr) * D + d, D, L > 0.f ? acc * (a.v_scale / L) : 0.f);
    } else {
      a.part_o[((head0 + hr) * a.nsplit + sp) * D + d] = acc;
      if (d == 0) a.part_ml[(head0 + hr) * a.nsplit + sp] = make_float2(L > 0.f ? M : -INFINITY, L);
    }
  }
}

// Merge of the splits of one (row, KV head) inside a thread-block cluster:
// every split left its (max, mass) pairs and unnormalised outputs in its own
// shared memory; the cluster's first CTA reads them through distributed
// shared memory, in split order, and writes the group's output.
template <int D>
__device__ __forceinline__ void merge_cluster(const AttnArgs& a, const float* qs, const float2* ml, int G,
                                              size_t head0, int ns) {
  for (int e = threadIdx.x; e < G * D; e += kAttnThreads) {
    const int hr = e / D, d = e - hr * D;
    // every split's (max, mass) and output first, all loads in flight at once
    float2 v[kAttnCluster];
    float ov[kAttnCluster];
#pragma unroll
    for (int sp = 0; sp < kAttnCluster; ++sp) {
      v[sp] = sp < ns ? ld_dsmem_f2(ml + hr, (uint32_t)sp) : make_float2(-INFINITY, 0.f);
      ov[sp] = sp < ns ? ld_dsmem_f32(qs + hr * D + d, (uint32_t)sp) : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < kAttnCluster; ++sp) if (v[sp].y > 0.f) M = fmaxf(M, v[sp].x);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int sp = 0; sp < kAttnCluster; ++sp) {
      if (v[sp].y > 0.f) {
        const float w = exp2f(v[sp].x - M);
        L += w * v[sp].y;
        acc += w * ov[sp];
      }
    }
    store_attn_out(a, (head0 + hr) * D + d, D, L > 0.f ? acc * (a.v_scale / L) : 0.f);
  }
}

// Merge the splits of the group's G query heads: rescale each partial to the
// common maximum, sum, divide by the total softmax mass, apply the V scale.
// Only the first na splits hold tokens (the others have zero mass). Their
// partials are pulled into shared memory with one round of cp.async per
// chunk (one L2 round trip instead of one per element a thread sums) while
// the (max, mass) pairs are read alongside; the weights then come from shared
// memory, one warp per head.
constexpr int kMergeMaxE = 16;     // G * D <= 16 * 128

__device__ __forceinline__ void merge_splits(const AttnArgs& a, unsigned char* smem, size_t smem_bytes, int G,
                                             size_t head0, int D, int na) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ns = a.nsplit;                                           // stride of the partials
  float2* sml = reinterpret_cast<float2*>(smem);                     // [G][na] (max, mass)
  float* wsm = reinterpret_cast<float*>(smem + (((size_t)G * na * 8 + 15) & ~(size_t)15));   // [G][na] weights
  const size_t w_bytes = (((size_t)G * na * 8 + 15) & ~(size_t)15) + (((size_t)G * na * 4 + 15) & ~(size_t)15);
  // running sums over chunks when the partials do not fit in one
  const bool one = w_bytes + (size_t)G * na * D * 4 <= smem_bytes;
  float* run = reinterpret_cast<float*>(smem + w_bytes);            // [G * D] (chunked only)
  float* so = one ? run : run + G * D;                               // [G][chunk][D]
  const size_t avail = smem_bytes - (size_t)((unsigned char*)so - smem);
  const int chunk = one ? na : max(1, (int)(avail / ((size_t)G * D * 4)));
  auto stage = [&](int s0, int sc) {
    const int per_g = sc * D / 4;                                    // float4 per head in this chunk
    for (int g = 0; g < G; ++g) {
      const float* src = a.part_o + ((head0 + g) * ns + s0) * D;
      float* dst = so + (size_t)g * sc * D;
      for (int j = tid; j < per_g; j += kAttnThreads) cp_async16(dst + 4 * j, src + 4 * j);
    }
    cp_async_commit();
  };
  stage(0, min(chunk, na));
  for (int i = tid; i < G * na; i += kAttnThreads) {
    const int g = i / na, sidx = i - g * na;
    sml[i] = a.part_ml[(head0 + g) * ns + sidx];
  }
  __syncthreads();                                                   // (max, mass) pairs staged
  for (int g = warp; g < G; g += kAttnThreads / 32) {
    const float2* ml = sml + g * na;
    float M = -INFINITY;
    for (int s = lane; s < na; s += 32) if (ml[s].y > 0.f) M = fmaxf(M, ml[s].x);
    M = warp_max(M);
    float L = 0.f;
    for (int s = lane; s < na; s += 32) if (ml[s].y > 0.f) L += exp2f(ml[s].x - M) * ml[s].y;
    L = warp_sum(L);
    const float inv = L > 0.f ? a.v_scale / L : 0.f;
    for (int s = lane; s < na; s += 32) wsm[g * na + s] = ml[s].y > 0.f ? exp2f(ml[s].x - M) * inv : 0.f;
  }
  for (int s0 = 0; s0 < na; s0 += chunk) {
    const int sc = min(chunk, na - s0);
    const bool last = s0 + chunk >= na;
    cp_async_wait<0>();
    __syncthreads();                                                 // chunk (and, first time, weights) ready
    for (int e = tid; e < G * D; e += kAttnThreads) {
      const int g = e / D, d = e - g * D;
      const float* po = so + (size_t)g * sc * D + d;
      const float* wg = wsm + g * na + s0;
      float acc0 = s0 ? run[e] : 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
      int s = 0;
      for (; s + 4 <= sc; s += 4) {
        const float w0 = wg[s], w1 = wg[s + 1], w2 = wg[s + 2], w3 = wg[s + 3];
        if (w0 != 0.f) acc0 += w0 * po[(size_t)s * D];
        if (w1 != 0.f) acc1 += w1 * po[(size_t)(s + 1) * D];
        if (w2 != 0.f) acc2 += w2 * po[(size_t)(s + 2) * D];
        if (w3 != 0.f) acc3 += w3 * po[(size_t)(s + 3) * D];
      }
    for (; s < sc; ++s) if (wg[s] != 0.f) acc0 += wg[s] * po[(size_t)s * D];
      const float o = (acc0 + acc1) + (acc2 + acc3);
      if (!last) { run[e] = o; continue; }
      store_attn_out(a, (head0 + g) * D + d, D, o);
    }
    if (!last) {
      __syncthreads();                                               // chunk consumed
      stage(s0 + chunk, min(chunk, na - s0 - chunk));
    }
  }
}

// One work item: split sp of the context of (row b, KV head h), and the merge
// of that group's splits when this is the last of them to finish.
template <int D, int KV8, int NT, int CL, int O4>
__device__ __forceinline__ void attn_item(const AttnArgs& a, unsigned char* smem, int sp, int h, int b) {
  using S = AttnShape<D, KV8, NT, O4>;
  const int G = a.nq / a.nkv;
  const int tid = threadIdx.x;
  const size_t head0 = (size_t)b * a.nq + (size_t)h * G;             // first query head of the group
  // step inputs (lengths, positions, block tables) are staged before the
  // step's first kernel starts, so they may be read before the wait
  const int seq = a.seq_lens[b];

  const bool seq_ok = seq >= 1 && seq <= a.bt_stride * kBlockTokens;
  if (!seq_ok && tid == 0 && sp == 0 && h == 0) set_err(a.err, MBT_DEV_SEQLEN_RANGE);
  const int nblk = seq_ok ? (seq + kBlockTokens - 1) / kBlockTokens : 0;
  const int blk0 = sp * a.bps;
  const int blk1 = min(nblk, blk0 + a.bps);

  // the split holding the new token's block writes its K and V
  bool writer = false;
  int pos = 0, wblk = 0;
  if (a.qkv) {
    pos = a.positions[b];
    const bool pos_ok = pos >= 0 && pos < a.max_pos;
    if (!pos_ok && tid == 0 && sp == 0 && h == 0) set_err(a.err, MBT_DEV_POS_RANGE);
    const int jb = pos_ok ? pos / kBlockTokens : -1;
    if (pos_ok && jb < a.bt_stride && sp == jb / a.bps) {
      wblk = a.bt[(size_t)b * a.bt_stride + jb];
      writer = wblk >= 0 && wblk <= a.num_blocks;
      if (!writer && tid == 0) set_err(a.err, MBT_DEV_BLOCK_RANGE);
    } else if (pos_ok && jb >= a.bt_stride && tid == 0 && sp == 0) {
      set_err(a.err, MBT_DEV_BLOCK_RANGE);
    }
  }

  __shared__ float2 cl_ml[16];                                        // cluster merge: (max, mass) per head
  if (blk0 < nblk) {
    attend<D, KV8, NT, CL, O4>(a, smem, b, h, sp, G, head0, seq, blk0, blk1, writer, pos, wblk, cl_ml);
  } else {
    pdl_wait();
    uint32_t kc, vc;
    if (writer) write_new_kv<D, KV8>(a, b, h, pos, wblk, kc, vc);
    if (CL) {
      if (tid < G) cl_ml[tid] = make_float2(-INFINITY, 0.f);
    } else if (a.nsplit == 1) {
      for (int e = tid; e < G * D; e += kAttnThreads) store_attn_out(a, head0 * D + e, D, 0.f);
    } else {
      if (tid < G) a.part_ml[(head0 + tid) * a.nsplit + sp] = make_float2(-INFINITY, 0.f);
    }
  }
  if (!CL && a.nsplit == 1) return;                                  // nothing to merge

  if (CL) {
    // the splits of this (row, KV head) are one cluster: merge through
    // distributed shared memory, then keep every CTA resident until the
    // merging CTA has read it
    cluster_sync_all();
    if (sp == 0) merge_cluster<D>(a, reinterpret_cast<const float*>(smem), cl_ml, G, head0, a.nsplit);
    cluster_sync_all();
    return;
  }

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
  // splits past the last one with tokens hold nothing to merge
  const int na = max(1, min(a.nsplit, (nblk + a.bps - 1) / a.bps));
  merge_splits(a, smem, S::SMEM, G, head0, D, na);
  if (tid == 0) a.tickets[(size_t)b * a.nkv + h] = 0;     // ready for the next launch
}

// One CTA per (split, KV head, row); the hardware hands out CTAs as earlier
// ones finish, which already balances splits of unequal length (a persistent
// grid claiming items from an atomic counter was measured slower: 91 vs 74 us
// per batch-64 8B-class layer).
template <int D, int KV8, int NT, int CL, int O4>
__global__ void __launch_bounds__(kAttnThreads, AttnShape<D, KV8, NT, O4>::MINB) attn_split_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_launch_dependents();
  attn_item<D, KV8, NT, CL, O4>(a, smem, blockIdx.x, blockIdx.y, blockIdx.z);
}

int attn_ctas_per_sm(int kv8, int G) { return kv8 && G <= 8 ? 4 : 3; }

void attn_plan(int B, int nkv, int max_blocks, int num_sms, int per_sm, int* bps, int* nsplit) {
  // Three CTAs per SM: about four CTAs per SM in all, so that rows with long
  // contexts do not form the tail (contexts in one batch differ by up to 8x).
  // Four per SM (e4m3 caches, up to 8 query heads): at most one wave, so that
  // batch 64 x 8 KV heads runs one split per (row, KV head) and needs no merge
  // (70B FP8 batch 64: 2.25 waves of two splits before). At least two 64-token
  // tiles per split either way, so that the copies overlap the math and the
  // merge stays short.
  const int pairs = B * nkv;
  int want = per_sm >= 4 ? 4 * num_sms / pairs : (4 * num_sms + pairs - 1) / pairs;
  if (want < 1) want = 1;
  int per = (max_blocks + want - 1) / want;
  const int min_per = MBT_ATTN_MIN_TILES * kAttnTile / kBlockTokens;
  if (per < min_per) per = min_per;
  if (per > max_blocks) per = max_blocks;
  // at most kAttnCluster splits, so that a (row, KV head) is one thread-block
  // cluster and its splits merge through distributed shared memory
  if (per < (max_blocks + kAttnCluster - 1) / kAttnCluster) per = (max_blocks + kAttnCluster - 1) / kAttnCluster;
  if (per > kMaxSplitBlocks) per = kMaxSplitBlocks;
  if (per < 1) per = 1;
  *bps = per;
  *nsplit = (max_blocks + per - 1) / per;
}

namespace {
template <int D, int KV8, int NT, int CL, int O4>
void* attn_fn() { return (void*)attn_split_kernel<D, KV8, NT, CL, O4>; }
// query heads per KV head: up to 8 in one n-tile of the MMA, up to 16 in two;
// cl: the splits of a (row, KV head) form one cluster; o4: the four-per-SM
// form (e4m3, one n-tile, no cluster)
template <int D, int KV8, int CL>
void* attn_fn_nt(int nt, int o4) {
  if (nt == 2) return attn_fn<D, KV8, 2, CL, 0>();
  return (KV8 && !CL && o4) ? attn_fn<D, KV8, 1, CL, 1>() : attn_fn<D, KV8, 1, CL, 0>();
}
template <int D, int KV8>
void* attn_fn_cl(int nt, int cl, int o4) { return cl ? attn_fn_nt<D, KV8, 1>(nt, 0) : attn_fn_nt<D, KV8, 0>(nt, o4); }
template <int D>
size_t attn_smem_of(int kv8, int nt, int o4) {
  if (kv8 && nt == 1 && o4) return AttnShape<D, 1, 1, 1>::SMEM;
  return kv8 ? (nt == 2 ? AttnShape<D, 1, 2>::SMEM : AttnShape<D, 1, 1>::SMEM)
             : (nt == 2 ? AttnShape<D, 0, 2>::SMEM : AttnShape<D, 0, 1>::SMEM);
}
void* attn_pick(int d, int kv8, int nt, int cl, int o4, size_t* smem) {
  o4 = o4 && kv8 && nt == 1 && !cl;
  if (d == 64) {
    *smem = attn_smem_of<64>(kv8, nt, o4);
    return kv8 ? attn_fn_cl<64, 1>(nt, cl, o4) : attn_fn_cl<64, 0>(nt, cl, o4);
  }
  *smem = attn_smem_of<128>(kv8, nt, o4);
  return kv8 ? attn_fn_cl<128, 1>(nt, cl, o4) : attn_fn_cl<128, 0>(nt, cl, o4);
}
}  // namespace

cudaError_t attn_init() {
  for (int d : {64, 128})
    for (int kv8 = 0; kv8 < 2; ++kv8)
      for (int nt = 1; nt <= 2; ++nt)
        for (int cl = 0; cl < 2; ++cl)
          for (int o4 = 0; o4 < 2; ++o4) {
            if (o4 && !(kv8 && nt == 1 && !cl)) continue;
            size_t sm;
            void* fn = attn_pick(d, kv8, nt, cl, o4, &sm);
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            // the four-per-SM form needs most of the unified L1 as shared memory
            if (e == cudaSuccess && o4) e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
            if (e != cudaSuccess) return e;
          }
  return cudaSuccess;
}

size_t attn_smem_bytes(int d, int kv8, int G) {
  size_t sm;
  attn_pick(d, kv8, G > 8 ? 2 : 1, 0, 0, &sm);            // the batch-1 form
  return sm + sizeof(int) * kMaxSplitBlocks + 16;     // + the staged block ids and the ticket flag
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s) {
  size_t sm;
  // the cluster merge pays off while the grid is about one wave (batch 1-4 at
  // 8 KV heads: 2.97 / 4.07 ms per 8B step); beyond that clusters of splits
  // packed the SMs worse than independent CTAs with the ticket merge (batch 8
  // and 16: 4.26 / 4.41 ms against 4.59 / 4.73 ms with clusters)
  static int nsm = 0;
  if (!nsm) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  }
  const int grid = a.B * a.nkv * a.nsplit;
  const int cl = a.nsplit >= 4 && a.nsplit <= kAttnCluster && grid <= 2 * nsm;
  // the four-per-SM e4m3 form once three per SM would not hold the grid in one wave
  const int o4 = grid > 3 * nsm;
  void* fn = attn_pick(a.d, a.kv_fp8, (a.nq / a.nkv) > 8 ? 2 : 1, cl, o4, &sm);
  // the merge needs the group's weights and at least one split of partials in shared memory
  const int G = a.nq / a.nkv;
  const size_t w_bytes = (((size_t)G * a.nsplit * 8 + 15) & ~(size_t)15) + (((size_t)G * a.nsplit * 4 + 15) & ~(size_t)15);
  if (G * a.d > kMergeMaxE * kAttnThreads || w_bytes + (size_t)2 * G * a.d * 4 > sm) return cudaErrorInvalidValue;
  AttnArgs args = a;
  void* params[] = {&args};
  return launch_ex(fn, dim3(a.nsplit, a.nkv, a.B), dim3(kAttnThreads), sm, s, params, !a.no_pdl,
                   a.carveout > 0 ? a.carveout : -1, cl ? a.nsplit : 0);
}

}  // namespace mbt
