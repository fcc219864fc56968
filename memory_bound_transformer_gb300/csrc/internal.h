// Launch interfaces between the runtime and the kernels (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace mbt {

typedef __nv_bfloat16 bf16;

enum Epilogue { EPI_PARTIAL = 0, EPI_SWIGLU = 1, EPI_ARGMAX = 2 };
enum Prologue { PRO_X = 0, PRO_NORM = 1 };

// Launch with the programmatic-stream-serialization attribute (PDL) so that the
// kernel's independent prologue overlaps the previous kernel's tail.
// Launch with programmatic dependent launch allowed (pdl = true) or as an
// ordinary stream-ordered launch; carveout >= 0 sets the shared-memory share
// of the unified L1 (percent) for this launch.
// cluster_x > 0: thread-block clusters of cluster_x CTAs along x
cudaError_t launch_ex(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args,
                      bool pdl, int carveout, int cluster_x = 0);
inline cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args,
                              int carveout = -1) {
  return launch_ex(fn, grid, block, smem, s, args, true, carveout);
}

struct ArgmaxPart { float v; int i; };

// Sampling draw fused into an arg-max epilogue: when `on`, the arg-max is taken
// over logit * inv_t + Gumbel(token, row0 + row, step; seed) instead of the
// logit (sampling.cuh); logits written out stay the raw ones.
struct GumbelArgs {
  int on; float inv_t; int row0;
  uint32_t seed_lo, seed_hi, step_lo, step_hi;
};

// y = W x for up to 8 batch rows (weight-streaming GEMV, CUDA cores).
// Shared-memory share of the unified L1 (percent) for every kernel of the
// CUDA-core (batch 1..15) step. Two things pull on it: the weight stream
// keeps ~128 KB of loads in flight per SM and those land in L1, so the
// share must stay well below the maximum; and neighbouring kernels overlap
// on an SM under programmatic dependent launch only if they ask for the same
// split (otherwise an SM drains before it takes the next kernel's CTAs).
// The model picks the smallest split that holds an attention CTA next to
// the O projection's GEMV CTA (stream_config); 44% = 100 KB suits an 8B-class
// model (measured on its batch-1 step: 44% 2.84 ms, 58% 2.89 ms, 72% 2.94 ms,
// 86-100% 3.45 ms) and is the default of the kernel-level entry points.
#ifndef MBT_SMEM_CARVEOUT
#define MBT_SMEM_CARVEOUT 44
#endif
#ifndef MBT_STREAM_SMEM_KB
#define MBT_STREAM_SMEM_KB 48
#endif
constexpr int kStreamCarveout = MBT_SMEM_CARVEOUT;
// largest dynamic shared memory of a GEMV CTA that runs two per SM under it
constexpr size_t kStreamSmemPerCta = (size_t)MBT_STREAM_SMEM_KB * 1024;
// Carveout (percent) and per-CTA GEMV shared-memory budget of one step.
struct StreamCfg {
  int carveout = kStreamCarveout;
  size_t cta_smem = kStreamSmemPerCta;
};
// The smallest supported split (100, 132, 164, 196 or 228 KB) that holds an
// attention CTA (attn_bytes, static + dynamic) next to a GEMV CTA whose x tile
// is o_k fp32 values, and the GEMV budget that lets two of those share an SM.
StreamCfg stream_config(size_t attn_bytes, int o_k);

struct GemvArgs {
  const void* W;            // [rows][K] row-major, BF16 or e4m3 codes
  const float* scale;       // per-row scale for e4m3 weights, else null
  int wtype;                // W_BF16 / W_E4M3
  int N;                    // output channels (SWIGLU: ffn; W holds 2N rows)
  int K;                    // multiple of 16
  const float* x; int ldx;  // PRO_X: [nb][ldx] fp32 input rows, 16-byte aligned
  int nb;                   // batch rows, 1..8
  // PRO_NORM: x = rmsnorm(r_in + sum_s delta[s]) * gamma over rows of K
  // elements; the CTA at (0, 0) stores r_in + sum_s delta[s] to r_out
  const float* r_in; const float* delta; int n_delta; long long delta_stride;
  const bf16* gamma; float eps; float* r_out;
  // EPI_PARTIAL: out[split * split_stride + b * ldo + n] (fp32, no accumulate)
  float* out; long long split_stride; int ldo;
  // EPI_SWIGLU: act[b * lda + n] = silu(gate_n) * up_n (fp32)
  float* act; int lda;
  // EPI_ARGMAX: per-CTA best (value, index) per row into part[cta * part_ld + b];
  // logits[b * ldl + n] written when logits != null
  float* logits; int ldl;
  ArgmaxPart* part; int part_ld;
  uint32_t* err;
  // bytes of this CTA's weight rows pulled into L2 before waiting on the
  // previous kernel (0 = default 64 KB); a kernel that follows a latency-bound
  // one (attention) prefetches its whole slice
  uint32_t prefetch_bytes;
  // Work queue for the tail (null: every CTA takes one fixed contiguous range
  // of rows). Otherwise CTA c first takes row groups [c*static_groups,
  // (c+1)*static_groups) and then claims the groups from grid*static_groups on,
  // one at a time, from the counter sched[split] (zero at launch; the CTA
  // that makes the last claim sets it back to zero).
  int* sched; int static_groups;
  GumbelArgs gum;           // EPI_ARGMAX: draw instead of arg-max when gum.on
};

struct GemvLaunch { int nb_tmpl; int nsplit; int grid; size_t smem; int group_rows; int carveout; };

// Static groups per CTA when this launch should take the work-queue tail
// (GemvArgs::sched, one zeroed counter per K split), else -1.
int gemv_queue_static_groups(const GemvLaunch& g, int N);

// Launch geometry for a GEMV of this shape (deterministic: the same inputs give
// the same geometry, so eager runs and graph replays do the same arithmetic).
GemvLaunch gemv_plan(int epi, int wtype, int nb, int N, int K, int num_sms, int force_nsplit,
                     int pro = PRO_X, const StreamCfg& sc = StreamCfg());
// Most batch rows one launch may take for this epilogue and prologue (the fp32
// x tile must fit in shared memory when K cannot be split).
int gemv_max_rows(int epi, int K, int pro = PRO_X);
cudaError_t gemv_launch(int epi, int pro, const GemvArgs& a, const GemvLaunch& g, cudaStream_t s);
cudaError_t gemv_init();   // raise dynamic shared-memory limits (once per process)

// Tensor-core skinny GEMMs (batch 2..128): y = W x. BF16 weights: x given as
// [2 * Rp][K] BF16 rows (rows 0..Rp-1 the high parts, Rp..2Rp-1 the low parts
// of the fp32 activations). e4m3 weights: x given as four e4m3 term rows
// [4][Rp][K] and one power-of-two scale per row (split_terms), multiplied
// e4m3 x e4m3. Tensor maps are opaque 128-byte blobs.
struct TmaMap { alignas(64) unsigned char bytes[128]; };
struct TcArgs {
  int N, K, R, Rp;            // output channels (SWIGLU: ffn), K, live rows of this launch, their padded count
  int row0, rp_all;           // first row of this launch; padded rows of the whole high/low buffer
  float* ts_scratch; int* ts_tickets; int tickets_cap;   // stream-K partial sums and per-tile tickets (zero)
  const float* scale;         // per-row weight scale or null
  float* out; long long split_stride; int ldo;       // EPI_PARTIAL: out[split][b][n]
  bf16* act_hl; int ld_act;                            // EPI_SWIGLU: [2 * Rp][ld_act] hi/lo rows
  int hl_f16;                                          // act_hl rows as FP16 (e4m3 weights), else BF16
  float* logits; int ldl; ArgmaxPart* part; int part_ld;   // EPI_ARGMAX
  uint32_t* err;
  GumbelArgs gum;                                      // EPI_ARGMAX: draw instead of arg-max when gum.on
  const float* x_scale;                                // e4m3 weights: the term rows' scales [rp_all]
};
cudaError_t tc_init();
cudaError_t tc_make_map(void* map, const void* base, int rows, int K, int box_rows);
// Stream-K tensor-core GEMM (tc_stream.cu): one CTA per SM, at most 64 rows
// (a.R <= a.Rp <= 64, a.Rp a multiple of 16) per launch; x as XR row blocks of
// [rp_all][K] (BF16 high then low rows; e4m3 terms 0..3, with a.x_scale), read
// from row a.row0 of each block with boxes of a.Rp rows. Outputs are complete
// sums (no K split): PARTIAL out[(row0 + b) * ldo + n].
cudaError_t ts_init();
cudaError_t ts_launch(int wt, int epi, const void* mapW, const void* mapX, const TcArgs& a, int num_sms,
                      cudaStream_t s);
int ts_tiles(int epi, int N);
size_t ts_scratch_floats(int num_sms);
constexpr int kTsMaxRows = 64;
// e4m3 codes [rows][K] (weights, with 64-row boxes, or activation term rows,
// with boxes of a launch's padded rows), 128-code boxes, 128-byte swizzle
cudaError_t tc_make_map_u8(void* map, const void* base, int rows, int K, int box_rows);
// fp32 rows x (or 16-bit high/low rows hl when x is null) -> term rows
// t [4][Rp][K] and scales ts[Rp]; rows B..Rp-1 zero with scale 1
cudaError_t tc_to_terms(const float* x, const bf16* hl, int f16, int B, int Rp, int K, uint8_t* t, float* ts,
                        cudaStream_t s);
cudaError_t tc_to_hl(const float* x, int B, int Rp, int K, bf16* hl, cudaStream_t s, int f16 = 0);
cudaError_t tc_from_hl(const bf16* hl, int B, int Rp, int N, float* out, cudaStream_t s, int f16 = 0);

// r <- E[token] (fp32); y <- rmsnorm(r) * gamma (fp32)
struct EmbedNormArgs {
  int B, H, vocab; const int* tokens; const bf16* embed;
  float* r; const bf16* gamma; float eps; float* y; uint32_t* err;
  int* zero; int n_zero;    // the step's GEMV work-queue counters, cleared here
  int carveout;             // launch carveout (percent); 0 (zero-initialised) = the default
};
cudaError_t launch_embed_rmsnorm(const EmbedNormArgs& a, cudaStream_t s);

// r <- r + sum_s delta[s]; y <- rmsnorm(r) * gamma (fp32), or, when y_hl is
// set, y as BF16 high/low rows [2 * rp][H] for the tensor-core GEMM (rows
// B..rp-1 written as zeros).
struct AddNormArgs {
  int B, H; float* r; const float* delta; int n_delta; long long delta_stride;
  const bf16* gamma; float eps; float* y;
  bf16* y_hl; int rp;
  int hl_f16;               // y_hl rows as FP16 (for e4m3 weights) rather than BF16
  // when set (and y_hl null): y as four e4m3 term rows [4][rp][H] with one
  // power-of-two scale per row, y_s[rp] (rows B..rp-1: zero codes, scale 1)
  uint8_t* y_t; float* y_s;
};
cudaError_t launch_add_rmsnorm(const AddNormArgs& a, cudaStream_t s);

// RoPE on q and k, q to q_out (fp32), k and v into the paged cache.
struct RopeKvArgs {
  int B; const float* qkv; int nsplit; long long split_stride; int ld_qkv;
  int nq, nkv, d; const int* positions; const int* bt; int bt_stride; int max_pos;
  const float2* rope;       // [max_pos][d/2] (cos, sin)
  float* q_out;             // [B][nq][d]
  void* kpool; void* vpool; // this layer's K and V pools [nb+1][nkv][16][d]
  int num_blocks;           // caller blocks; id num_blocks = null block
  int kv_fp8; float k_scale, v_scale; uint32_t* err;
};
cudaError_t launch_rope_kv_write(const RopeKvArgs& a, cudaStream_t s);

// Split-K paged decode attention; the last CTA of each (row, KV head) merges
// the splits (ticket counters in `tickets`, zero between launches).
struct AttnArgs {
  int B; const float* q; int nq, nkv, d;
  // Fused RoPE + KV write (when qkv != null, q is ignored): the queries are
  // rotated from the QKV projection's split-K partials in the prologue, and the
  // CTA whose split holds the new token's block first writes its K and V.
  const float* qkv; int qkv_nsplit; long long qkv_split_stride; int ld_qkv;
  const int* positions; const float2* rope; int max_pos;
  const void* kpool; const void* vpool; int kv_fp8; float k_scale, v_scale;
  const int* bt; int bt_stride; const int* seq_lens; int num_blocks;
  int bps; int nsplit;      // KV blocks per split, splits per (row, kv head)
  float* part_o; float2* part_ml; float* out; int* tickets; uint32_t* err;
  bf16* out_hl; int rp_hl;  // optional: output also as 16-bit high/low rows [2 * rp_hl][nq * d]
  int hl_f16;               // out_hl as FP16 (for e4m3 weights) rather than BF16
  int carveout;             // launch carveout (percent); 0 (zero-initialised) = the default
  int no_pdl;               // ordinary launch: the previous kernel wrote this layer's cache
};
// CTAs of the attention kernel resident per SM (3, or 4 for e4m3 caches with
// up to 8 query heads per KV head), the input of attn_plan's wave sizing.
int attn_ctas_per_sm(int kv8, int G);
void attn_plan(int B, int nkv, int max_blocks, int num_sms, int per_sm, int* bps, int* nsplit);
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s);
cudaError_t attn_init();
size_t attn_smem_bytes(int d, int kv8, int G);   // static + dynamic shared memory of one attention CTA

// next_ids[b] = index of the best of part[0..G)[b]
cudaError_t launch_argmax_reduce(int B, const ArgmaxPart* part, int part_ld, int G,
                                 int* next_ids, uint32_t* err, cudaStream_t s, int carveout = -1);

// Top-k / top-p draw per row from logits in memory (rows of ldl floats): the
// k largest logit * inv_t (ties: lower id), softmax over them, the shortest
// most-probable prefix reaching top_p, and the Gumbel-max draw over it.
// k in 1..kTopKMax.
constexpr int kTopKMax = 1024;
struct TopKArgs {
  int B, V, ldl; const float* logits; float inv_t; int k; float top_p;
  GumbelArgs gum; int* next_ids; uint32_t* err;
};
cudaError_t launch_sample_topk(const TopKArgs& a, cudaStream_t s);

// Copy B caller rows into the graph's static buffers and fill pad rows [B, R).
// Live rows keep the caller's table width: entries from bt_stride on are
// written as -1 (an invalid id), and a row whose seq_len needs more than
// bt_stride blocks gets seq_len 0 and MBT_DEV_SEQLEN_RANGE in err, so the
// graph treats it as the eager path does (no attention, error bit set).
struct StageArgs {
  int B, R; const int* tok; const int* pos; const int* bt; int bt_stride; const int* sl;
  int* s_tok; int* s_pos; int* s_bt; int s_stride; int* s_sl; int null_block;
  uint32_t* err;
};
cudaError_t launch_stage_inputs(const StageArgs& a, cudaStream_t s);

// Rows of one prefill pass: R consecutive prompt tokens of one sequence from
// position p0 on (token, position, seq_len = position + 1, and the
// sequence's block table repeated per row).
struct PrefillStageArgs {
  int R; const int* tokens; int p0; const int* bt; int bt_len;
  int* s_tok; int* s_pos; int* s_sl; int* s_bt;
};
cudaError_t launch_stage_prefill(const PrefillStageArgs& a, cudaStream_t s);

}  // namespace mbt
