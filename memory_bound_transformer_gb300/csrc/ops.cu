// Kernel-level entry points (include/mbt_ops.h): one decode-step kernel per
// call on caller buffers, with the decode step's launch geometry.
#include <algorithm>
#include <cmath>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "../../include/mbt_ops.h"

using namespace mbt;

namespace {
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}
bool inited = false;
int init_once() {
  if (inited) return MBT_OK;
  if (gemv_init() != cudaSuccess || attn_init() != cudaSuccess) return MBT_ERR_CUDA;
  inited = true;
  return MBT_OK;
}
}  // namespace

extern "C" {

int op_embed_rmsnorm(int B, int H, int vocab, const int32_t* tokens, const uint16_t* embed,
                     const uint16_t* gamma, float eps, float* r, float* y, uint32_t* err,
                     void* stream) {
  if (B < 1 || H < 4 || H % 4 || vocab < 1 || !tokens || !embed || !gamma || !r || !y) return MBT_ERR_BAD_ARG;
  EmbedNormArgs a{B, H, vocab, tokens, (const bf16*)embed, r, (const bf16*)gamma, eps, y, err};
  return launch_embed_rmsnorm(a, (cudaStream_t)stream) == cudaSuccess ? MBT_OK : MBT_ERR_CUDA;
}

int op_add_rmsnorm(int B, int H, float* r, const float* delta, int n_delta,
                   const uint16_t* gamma, float eps, float* y, void* stream) {
  if (B < 1 || H < 4 || H % 4 || !r || !gamma || !y || n_delta < 0 || (n_delta && !delta)) return MBT_ERR_BAD_ARG;
  AddNormArgs a{B, H, r, delta, n_delta, (long long)B * H, (const bf16*)gamma, eps, y, nullptr, 0};
  return launch_add_rmsnorm(a, (cudaStream_t)stream) == cudaSuccess ? MBT_OK : MBT_ERR_CUDA;
}

int op_gemv_nsplit(int epi, int w_dtype, int B, int N, int K) {
  const int n = sm_count();
  if (n <= 0 || B < 1 || N < 1 || K < 16) return 1;
  return gemv_plan(epi, w_dtype == MBT_DTYPE_E4M3 ? W_E4M3 : W_BF16, std::min(B, 8), N, K, n, 0).nsplit;
}

int op_gemv(int epi, int w_dtype, const void* W, const float* scales, int N, int K,
            const float* x, int B, int force_nsplit, float* out, float* act,
            float* logits, int32_t* next_ids, int* nsplit_used, uint32_t* err, void* stream) {
  return op_gemv_ex(epi, w_dtype, W, scales, N, K, x, B, force_nsplit, out, act, logits, next_ids,
                    nsplit_used, nullptr, err, stream);
}

int op_gemv_sched_ints(int epi, int w_dtype, int B, int N, int K) {
  const int n = sm_count();
  if (n <= 0 || B < 1 || N < 1 || K < 16) return 0;
  const int step = gemv_max_rows(epi, K);
  const GemvLaunch g = gemv_plan(epi, w_dtype == MBT_DTYPE_E4M3 ? W_E4M3 : W_BF16, std::min(B, step), N, K, n, 0);
  return ((B + step - 1) / step) * g.nsplit;
}

}  // extern "C"

namespace {
// The step's residual-add + RMSNorm prologue inputs (null: x is given).
struct NormOp { const float* r_in; const float* delta; int n_delta; const uint16_t* gamma; float eps; float* r_out; };

int gemv_impl(int epi, int w_dtype, const void* W, const float* scales, int N, int K, const float* x,
              const NormOp* nin, int B, int force_nsplit, float* out, float* act, float* logits,
              int32_t* next_ids, int* nsplit_used, int* sched_ints, uint32_t* err, void* stream) {
  if (epi < 0 || epi > 2 || (w_dtype != MBT_DTYPE_BF16 && w_dtype != MBT_DTYPE_E4M3)) return MBT_ERR_BAD_ARG;
  if (!W || (!x && !nin) || B < 1 || N < 1 || K < 16 || K % 16) return MBT_ERR_BAD_ARG;
  if (nin && (!nin->r_in || !nin->gamma || !nin->r_out || nin->n_delta < 0 || (nin->n_delta && !nin->delta)))
    return MBT_ERR_BAD_ARG;
  if (w_dtype == MBT_DTYPE_E4M3 && !scales) return MBT_ERR_BAD_ARG;
  if ((epi == EPI_PARTIAL && !out) || (epi == EPI_SWIGLU && !act) || (epi == EPI_ARGMAX && !next_ids))
    return MBT_ERR_BAD_ARG;
  int rc = init_once();
  if (rc != MBT_OK) return rc;
  const int nsm = sm_count();
  const int wt = w_dtype == MBT_DTYPE_E4M3 ? W_E4M3 : W_BF16;
  const int pro = nin ? PRO_NORM : PRO_X;
  cudaStream_t s = (cudaStream_t)stream;
  const int step = gemv_max_rows(epi, K, pro);
  const GemvLaunch g0 = gemv_plan(epi, wt, std::min(B, step), N, K, nsm,
                                  epi == EPI_PARTIAL ? force_nsplit : 0, pro);
  if (nsplit_used) *nsplit_used = g0.nsplit;
  ArgmaxPart* part = nullptr;
  if (epi == EPI_ARGMAX &&
      cudaMallocAsync((void**)&part, (size_t)g0.grid * B * sizeof(ArgmaxPart), s) != cudaSuccess)
    return MBT_ERR_OOM;
  // work-queue counters, one per launch and K split, zero at launch (the
  // kernel leaves them at zero): the caller's, or allocated and zeroed here
  const int nlaunch = (B + step - 1) / step;
  int* sched = sched_ints;
  bool own = false;
  if (!sched && gemv_queue_static_groups(g0, N) >= 0) {
    const size_t bytes = (size_t)nlaunch * g0.nsplit * sizeof(int);
    if (cudaMallocAsync((void**)&sched, bytes, s) != cudaSuccess) {
      if (part) cudaFreeAsync(part, s);
      return MBT_ERR_OOM;
    }
    own = true;
    if (cudaMemsetAsync(sched, 0, bytes, s) != cudaSuccess) rc = MBT_ERR_CUDA;
  }
  for (int b0 = 0; b0 < B && rc == MBT_OK; b0 += step) {
    const int nb = std::min(step, B - b0);
    GemvLaunch g = gemv_plan(epi, wt, nb, N, K, nsm, epi == EPI_PARTIAL ? g0.nsplit : 0, pro);
    if (epi == EPI_ARGMAX) g.grid = g0.grid;
    GemvArgs a = {};
    a.W = W; a.scale = scales; a.wtype = wt; a.N = N; a.K = K;
    a.x = x ? x + (size_t)b0 * K : nullptr; a.ldx = K; a.nb = nb;
    if (nin) {
      a.r_in = nin->r_in + (size_t)b0 * K;
      a.delta = nin->delta ? nin->delta + (size_t)b0 * K : nullptr;
      a.n_delta = nin->n_delta; a.delta_stride = (long long)B * K;
      a.gamma = (const bf16*)nin->gamma; a.eps = nin->eps;
      a.r_out = nin->r_out + (size_t)b0 * K;
    }
    a.out = out ? out + (size_t)b0 * N : nullptr; a.split_stride = (long long)B * N; a.ldo = N;
    a.act = act ? act + (size_t)b0 * N : nullptr; a.lda = N;
    a.logits = logits ? logits + (size_t)b0 * N : nullptr; a.ldl = N;
    a.part = part ? part + b0 : nullptr; a.part_ld = B;
    a.err = err;
    const int sg = gemv_queue_static_groups(g, N);
    if (sched && sg >= 0) {
      a.sched = sched + (size_t)(b0 / step) * g0.nsplit;
      a.static_groups = sg;
    }
    if (gemv_launch(epi, pro, a, g, s) != cudaSuccess) rc = MBT_ERR_CUDA;
  }
  if (rc == MBT_OK && epi == EPI_ARGMAX &&
      launch_argmax_reduce(B, part, B, g0.grid, next_ids, err, s) != cudaSuccess)
    rc = MBT_ERR_CUDA;
  if (part) cudaFreeAsync(part, s);
  if (own) cudaFreeAsync(sched, s);
  return rc;
}
}  // namespace

extern "C" {

int op_gemv_ex(int epi, int w_dtype, const void* W, const float* scales, int N, int K,
               const float* x, int B, int force_nsplit, float* out, float* act,
               float* logits, int32_t* next_ids, int* nsplit_used, int* sched_ints, uint32_t* err,
               void* stream) {
  return gemv_impl(epi, w_dtype, W, scales, N, K, x, nullptr, B, force_nsplit, out, act, logits, next_ids,
                   nsplit_used, sched_ints, err, stream);
}

int op_gemv_norm_sched_ints(int epi, int w_dtype, int B, int N, int K) {
  const int n = sm_count();
  if (n <= 0 || B < 1 || N < 1 || K < 16) return 0;
  const int step = gemv_max_rows(epi, K, PRO_NORM);
  const GemvLaunch g = gemv_plan(epi, w_dtype == MBT_DTYPE_E4M3 ? W_E4M3 : W_BF16, std::min(B, step), N, K, n, 0,
                                 PRO_NORM);
  return ((B + step - 1) / step) * g.nsplit;
}

int op_gemv_norm(int epi, int w_dtype, const void* W, const float* scales, int N, int K,
                 const float* r_in, const float* delta, int n_delta, const uint16_t* gamma, float eps,
                 float* r_out, int B, float* out, float* act, float* logits, int32_t* next_ids,
                 int* sched_ints, uint32_t* err, void* stream) {
  const NormOp nin{r_in, delta, n_delta, gamma, eps, r_out};
  return gemv_impl(epi, w_dtype, W, scales, N, K, nullptr, &nin, B, 0, out, act, logits, next_ids, nullptr,
                   sched_ints, err, stream);
}

namespace {
// Shared body of the BF16 (f8 = 0) and e4m3 (f8 = 1) tensor-core entry points:
// x split into BF16 high/low rows (BF16 weights) or e4m3 term rows and row
// scales (e4m3 weights), the stream-K GEMM in launches of at most 64 rows (the
// decode step's geometry), SwiGLU rows (16-bit high/low) read back to fp32.
int gemm_tc_impl(int f8, int epi, const void* W, const float* scales, int N, int K, const float* x, int B,
                 int ksplit, float* out, float* act, float* logits, int32_t* next_ids, uint32_t* err,
                 void* stream) {
  (void)ksplit;                                  // complete sums: the GEMM splits K across CTAs itself
  if (f8 && !scales) return MBT_ERR_BAD_ARG;
  if (epi < 0 || epi > 2 || !W || !x || B < 1 || B > 128 || N < 1 || K < 64 || K % 16) return MBT_ERR_BAD_ARG;
  if ((epi == EPI_PARTIAL && !out) || (epi == EPI_SWIGLU && !act) || (epi == EPI_ARGMAX && !next_ids))
    return MBT_ERR_BAD_ARG;
  {
    cudaError_t e = tc_init();
    if (e == cudaErrorNotSupported) return MBT_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return MBT_ERR_CUDA;
  }
  int rc = init_once();
  if (rc != MBT_OK) return rc;
  const int nsm = sm_count();
  cudaStream_t s = (cudaStream_t)stream;
  const int Rp = (B + 15) / 16 * 16;
  const int wrows = epi == EPI_SWIGLU ? 2 * N : N;
  const int tiles = ts_tiles(epi, N);
  const size_t b_x = (size_t)2 * Rp * K * 2 + (size_t)Rp * 4, b_a = epi == EPI_SWIGLU ? (size_t)2 * Rp * N * 2 : 0;
  const size_t b_p = epi == EPI_ARGMAX ? (size_t)tiles * B * sizeof(ArgmaxPart) : 0;
  const size_t b_s = ts_scratch_floats(nsm) * 4, b_t = (size_t)tiles * 4;
  auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
  char* scratch = nullptr;
  if (cudaMallocAsync((void**)&scratch, al(b_x) + al(b_a) + al(b_p) + al(b_s) + al(b_t), s) != cudaSuccess)
    return MBT_ERR_OOM;
  bf16* xhl = (bf16*)scratch;                    // BF16 high/low rows, or e4m3 term rows (same bytes)
  float* xsc = (float*)(scratch + (size_t)2 * Rp * K * 2);
  bf16* ahl = (bf16*)(scratch + al(b_x));
  ArgmaxPart* part = (ArgmaxPart*)((char*)ahl + al(b_a));
  float* tss = (float*)((char*)part + al(b_p));
  int* tickets = (int*)((char*)tss + al(b_s));
  TmaMap wm;
  const cudaError_t me = f8 ? tc_make_map_u8(&wm, W, wrows, K, 64) : tc_make_map(&wm, W, wrows, K, 64);
  if (me != cudaSuccess) rc = MBT_ERR_BAD_ARG;
  if (rc == MBT_OK && cudaMemsetAsync(tickets, 0, b_t, s) != cudaSuccess) rc = MBT_ERR_CUDA;
  if (rc == MBT_OK) {
    const cudaError_t e = f8 ? tc_to_terms(x, nullptr, 0, B, Rp, K, (uint8_t*)xhl, xsc, s) : tc_to_hl(x, B, Rp, K, xhl, s, 0);
    if (e != cudaSuccess) rc = MBT_ERR_CUDA;
  }
  for (int r0 = 0; r0 < B && rc == MBT_OK; r0 += kTsMaxRows) {
    const int rl = std::min(kTsMaxRows, B - r0), rcp = (rl + 15) / 16 * 16;
    TmaMap xm;
    const cudaError_t xe = f8 ? tc_make_map_u8(&xm, xhl, kTerms * Rp, K, rcp) : tc_make_map(&xm, xhl, 2 * Rp, K, rcp);
    if (xe != cudaSuccess) { rc = MBT_ERR_BAD_ARG; break; }
    TcArgs a = {};
    a.N = N; a.K = K; a.R = rl; a.Rp = rcp; a.row0 = r0; a.rp_all = Rp; a.scale = scales;
    a.out = out; a.split_stride = (long long)B * N; a.ldo = N;
    a.act_hl = ahl; a.ld_act = N; a.hl_f16 = f8; a.x_scale = f8 ? xsc : nullptr;
    a.logits = logits; a.ldl = N; a.part = part; a.part_ld = B; a.err = err;
    a.ts_scratch = tss; a.ts_tickets = tickets; a.tickets_cap = tiles;
    if (ts_launch(f8 ? W_E4M3 : W_BF16, epi, &wm, &xm, a, nsm, s) != cudaSuccess) rc = MBT_ERR_CUDA;
  }
  if (rc == MBT_OK && epi == EPI_SWIGLU && tc_from_hl(ahl, B, Rp, N, act, s, f8) != cudaSuccess) rc = MBT_ERR_CUDA;
  if (rc == MBT_OK && epi == EPI_ARGMAX && launch_argmax_reduce(B, part, B, tiles, next_ids, err, s) != cudaSuccess)
    rc = MBT_ERR_CUDA;
  cudaFreeAsync(scratch, s);
  return rc;
}
}  // namespace

int op_gemm_tc(int epi, const void* W, const float* scales, int N, int K, const float* x, int B,
               int ksplit, float* out, float* act, float* logits, int32_t* next_ids, uint32_t* err,
               void* stream) {
  return gemm_tc_impl(0, epi, W, scales, N, K, x, B, ksplit, out, act, logits, next_ids, err, stream);
}

int op_gemm_tc_e4m3(int epi, const void* W, const float* scales, int N, int K, const float* x, int B,
                    int ksplit, float* out, float* act, float* logits, int32_t* next_ids, uint32_t* err,
                    void* stream) {
  return gemm_tc_impl(1, epi, W, scales, N, K, x, B, ksplit, out, act, logits, next_ids, err, stream);
}

int op_rope_kv_write(int B, const float* qkv, int nq, int nkv, int d, const int32_t* positions,
                     const int32_t* bt, int bt_stride, int max_pos, float theta, void* kpool,
                     void* vpool, int num_blocks, int kv_dtype, float k_scale, float v_scale,
                     float* q_out, uint32_t* err, void* stream) {
  if (B < 1 || !qkv || nq < 1 || nkv < 1 || (d != 64 && d != 128) || !positions || !bt ||
      bt_stride < 1 || max_pos < 1 || !kpool || !vpool || num_blocks < 1 || !q_out ||
      !(k_scale > 0.f) || !(v_scale > 0.f) || (kv_dtype != MBT_DTYPE_BF16 && kv_dtype != MBT_DTYPE_E4M3))
    return MBT_ERR_BAD_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int half = d / 2;
  std::vector<float2> tab((size_t)max_pos * half);
  for (int p = 0; p < max_pos; ++p)
    for (int i = 0; i < half; ++i) {
      const double ang = (double)p * std::pow((double)theta, -2.0 * i / (double)d);
      tab[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
  float2* rope = nullptr;
  if (cudaMallocAsync((void**)&rope, tab.size() * sizeof(float2), s) != cudaSuccess) return MBT_ERR_OOM;
  int rc = MBT_OK;
  if (cudaMemcpyAsync(rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice, s) != cudaSuccess)
    rc = MBT_ERR_CUDA;
  RopeKvArgs a = {};
  a.B = B; a.qkv = qkv; a.nsplit = 1; a.split_stride = 0; a.ld_qkv = (nq + 2 * nkv) * d;
  a.nq = nq; a.nkv = nkv; a.d = d; a.positions = positions; a.bt = bt; a.bt_stride = bt_stride;
  a.max_pos = max_pos; a.rope = rope; a.q_out = q_out; a.kpool = kpool; a.vpool = vpool;
  a.num_blocks = num_blocks; a.kv_fp8 = kv_dtype == MBT_DTYPE_E4M3; a.k_scale = k_scale;
  a.v_scale = v_scale; a.err = err;
  if (rc == MBT_OK && launch_rope_kv_write(a, s) != cudaSuccess) rc = MBT_ERR_CUDA;
  // the table must outlive the kernel: free in stream order, then wait for the
  // host vector's copy to finish before it goes out of scope
  cudaFreeAsync(rope, s);
  if (cudaStreamSynchronize(s) != cudaSuccess) rc = MBT_ERR_CUDA;
  return rc;
}

int op_paged_attention(int B, const float* q, int nq, int nkv, int d, const void* kpool,
                       const void* vpool, int kv_dtype, float k_scale, float v_scale,
                       const int32_t* bt, int bt_stride, const int32_t* seq_lens, int num_blocks,
                       float* out, uint32_t* err, void* stream) {
  if (B < 1 || !q || nq < 1 || nkv < 1 || nq % nkv || nq / nkv > 16 || (d != 64 && d != 128) ||
      !kpool || !vpool || !bt || bt_stride < 1 || !seq_lens || num_blocks < 1 || !out ||
      (kv_dtype != MBT_DTYPE_BF16 && kv_dtype != MBT_DTYPE_E4M3))
    return MBT_ERR_BAD_ARG;
  int rc = init_once();
  if (rc != MBT_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  AttnArgs a = {};
  a.B = B; a.q = q; a.nq = nq; a.nkv = nkv; a.d = d; a.kpool = kpool; a.vpool = vpool;
  a.kv_fp8 = kv_dtype == MBT_DTYPE_E4M3; a.k_scale = k_scale; a.v_scale = v_scale;
  a.bt = bt; a.bt_stride = bt_stride; a.seq_lens = seq_lens; a.num_blocks = num_blocks;
  attn_plan(B, nkv, bt_stride, sm_count(), attn_ctas_per_sm(a.kv_fp8, nq / nkv), &a.bps, &a.nsplit);
  a.out = out; a.err = err;
  const size_t heads = (size_t)B * nq * a.nsplit;
  // scratch: partial outputs, (max, sum) pairs, zeroed tickets
  const size_t b_po = heads * d * sizeof(float), b_ml = heads * sizeof(float2);
  const size_t b_tk = (size_t)B * nkv * sizeof(int);
  char* scratch = nullptr;
  if (cudaMallocAsync((void**)&scratch, b_po + b_ml + b_tk, s) != cudaSuccess) return MBT_ERR_OOM;
  a.part_o = (float*)scratch;
  a.part_ml = (float2*)(scratch + b_po);
  a.tickets = (int*)(scratch + b_po + b_ml);
  if (cudaMemsetAsync(a.tickets, 0, b_tk, s) != cudaSuccess) rc = MBT_ERR_CUDA;
  if (rc == MBT_OK && launch_attention(a, s) != cudaSuccess) rc = MBT_ERR_CUDA;
  cudaFreeAsync(scratch, s);
  return rc;
}

}  // extern "C"
