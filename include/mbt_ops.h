/*
 * mbt_ops.h -- kernel-level entry points of libmbt.so.
 *
 * Each call runs one kernel of the decode step (the same kernel and launch
 * geometry the step uses) on caller buffers, so that every stage can be checked
 * on its own at full model sizes. Conventions are those of mbt.h: 0 on success,
 * negative MBT_ERR_* codes, device pointers in CUDA device memory, asynchronous
 * on `stream`. Calls that need scratch space take it from the stream-ordered
 * allocator (cudaMallocAsync / cudaFreeAsync on `stream`). `err` is a device
 * uint32 the kernels OR MBT_DEV_* bits into (may be NULL).
 * BF16 arrays (weights, gains) are passed as uint16 bit patterns; activations
 * are fp32.
 */
#ifndef MBT_OPS_H_
#define MBT_OPS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MBT_EPI_PARTIAL 0   /* fp32 split-K partial sums out[split][B][N]              */
#define MBT_EPI_SWIGLU  1   /* act[B][N] = silu(gate) * up (fp32), W has 2N rows       */
#define MBT_EPI_ARGMAX  2   /* next_ids[B] = argmax_n (W x)_n, logits[B][N] if non-NULL */

/* op_embed_rmsnorm: r[b] = E[tokens[b]] (fp32), y[b] = r / sqrt(mean(r^2) + eps)
 * * gamma (fp32). RMSNorm as defined in "Root Mean Square Layer
 * Normalization" (reference 9 of "Kernel Fusion for Large-Scale LLM
 * Inference"). embed [vocab][H] and gamma [H] BF16; r, y [B][H] fp32; H a
 * multiple of 4. */
int op_embed_rmsnorm(int B, int H, int vocab, const int32_t* tokens, const uint16_t* embed,
                     const uint16_t* gamma, float eps, float* r, float* y, uint32_t* err,
                     void* stream);

/* op_add_rmsnorm: r[b] += sum_s delta[s][b]; y[b] = rmsnorm(r[b]) * gamma
 * ("Kernels, Fusion & CUDA Graphs", "Fix 1: kernel fusion": residual add +
 * RMSNorm in one pass). delta [n_delta][B][H] fp32 (n_delta may be 0); r, y
 * fp32; gamma BF16. */
int op_add_rmsnorm(int B, int H, float* r, const float* delta, int n_delta,
                   const uint16_t* gamma, float eps, float* y, void* stream);

/* op_gemv_nsplit: split-K count op_gemv uses for this shape (1 unless PARTIAL). */
int op_gemv_nsplit(int epi, int w_dtype, int B, int N, int K);

/* op_gemv: the weight-streaming projection for B rows (any B >= 1; rows are
 * processed 8 at a time). W [rows][K] row-major, BF16 or e4m3 codes (w_dtype
 * MBT_DTYPE_BF16 / MBT_DTYPE_E4M3) with fp32 per-row scales (NULL for BF16);
 * x [B][K] fp32; K a multiple of 16.
 *   PARTIAL: out [nsplit][B][N] fp32, nsplit = op_gemv_nsplit(...) unless
 *            force_nsplit > 0 (clamped to K / 8 for BF16, K / 16 for e4m3);
 *            *nsplit_used receives it (may be NULL).
 *   SWIGLU:  W has 2N rows (gate rows then up rows); act [B][N] fp32.
 *   ARGMAX:  next_ids [B] int32; logits [B][N] fp32 or NULL.
 * Dequantisation is fused into the projection ("Kernel Fusion for Large-Scale
 * LLM Inference", section 11, "Epilogue and dequant fusion"). */
int op_gemv(int epi, int w_dtype, const void* W, const float* scales, int N, int K,
            const float* x, int B, int force_nsplit, float* out, float* act,
            float* logits, int32_t* next_ids, int* nsplit_used, uint32_t* err, void* stream);

/* op_gemv_sched_ints: ints of work-queue counters op_gemv_ex may use for this
 * shape (the projections split their tail into row groups claimed at run
 * time from one counter per launch and K split). */
int op_gemv_sched_ints(int epi, int w_dtype, int B, int N, int K);

/* op_gemv_ex: op_gemv with caller-owned work-queue counters: sched_ints
 * (device, op_gemv_sched_ints(...) ints) must be zero when the call is issued
 * and is zero again when it completes, so one array serves any number of
 * calls issued in order on one stream (not calls that run concurrently).
 * NULL: the counters are allocated and zeroed per call, as op_gemv does. The
 * pages have no counterpart: it exists so that back-to-back launches (timing
 * one projection, for one) carry no memset between them. */
int op_gemv_ex(int epi, int w_dtype, const void* W, const float* scales, int N, int K,
               const float* x, int B, int force_nsplit, float* out, float* act,
               float* logits, int32_t* next_ids, int* nsplit_used, int* sched_ints, uint32_t* err,
               void* stream);

/* op_gemv_norm_sched_ints: ints of work-queue counters op_gemv_norm may use. */
int op_gemv_norm_sched_ints(int epi, int w_dtype, int B, int N, int K);

/* op_gemv_norm: the projection as the decode step launches it at batch 1..15,
 * with the residual add + RMSNorm as its prologue ("Kernels, Fusion & CUDA
 * Graphs", "Fix 1: kernel fusion": residual add + RMSNorm in one pass, fused
 * here into the projection that consumes it): every CTA forms
 * x[b] = rmsnorm(r_in[b] + sum_s delta[s][b]) * gamma into its own tile and
 * the call stores the new residual r_in[b] + sum_s delta[s][b] to r_out[b].
 * r_in, r_out [B][K] fp32 (distinct buffers); delta [n_delta][B][K] fp32 or
 * NULL with n_delta = 0; gamma [K] BF16; eps inside the square root. No K
 * split: PARTIAL writes out [1][B][N]. Other arguments as op_gemv_ex
 * (sched_ints from op_gemv_norm_sched_ints, or NULL). Launch geometry and
 * shared-memory carveout are those of an 8B-class model's step. */
int op_gemv_norm(int epi, int w_dtype, const void* W, const float* scales, int N, int K,
                 const float* r_in, const float* delta, int n_delta, const uint16_t* gamma, float eps,
                 float* r_out, int B, float* out, float* act, float* logits, int32_t* next_ids,
                 int* sched_ints, uint32_t* err, void* stream);

/* op_gemm_tc: the tensor-core (tcgen05) projection the decode step uses from
 * 2 rows on with BF16 weights: W [rows][K] BF16 (K a multiple of 16, >= 64),
 * x [B][K] fp32 with 1 <= B <= 128, split internally into BF16 high/low rows
 * so that the product keeps near-fp32 accuracy; launches of at most 64 rows,
 * each CTA taking an equal share of the (tile, K) work and the fp32 sums kept
 * in registers. Epilogues as op_gemv: PARTIAL out [B][N] (complete sums:
 * `ksplit` is accepted and ignored), SWIGLU act [B][N] fp32 (W has 2N rows),
 * ARGMAX next_ids [B] (+ logits [B][N] if non-NULL). Returns
 * MBT_ERR_UNSUPPORTED where the tensor-map encoder is unavailable. ("GPU
 * Inference Internals", "Roofline: Why Decode Is Memory-Bound": at batch B the
 * weight-only intensity is 2B / b_w FLOP per byte.) */
int op_gemm_tc(int epi, const void* W, const float* scales, int N, int K, const float* x, int B,
               int ksplit, float* out, float* act, float* logits, int32_t* next_ids, uint32_t* err,
               void* stream);

/* op_gemm_tc_e4m3: as op_gemm_tc for e4m3 weights W [rows][K] (codes) with
 * fp32 per-row scales (required): x is split internally into four e4m3 terms
 * per value with a power-of-two scale per row (x = s (c0 + c1/16 + c2/256 +
 * c3/4096), within 2^-16 of |x| plus 2^-29 of the row's largest value), the
 * codes are multiplied as they are (e4m3 x e4m3 products, fp32 sums), and the
 * row scales are applied in the epilogue ("Kernel Fusion for Large-Scale LLM
 * Inference", section 11, FP8 weights and "Epilogue and dequant fusion"). The
 * SWIGLU rows pass through FP16 high/low pairs before act. K a multiple of 16,
 * >= 64; 1 <= B <= 128. */
int op_gemm_tc_e4m3(int epi, const void* W, const float* scales, int N, int K, const float* x, int B,
                    int ksplit, float* out, float* act, float* logits, int32_t* next_ids, uint32_t* err,
                    void* stream);

/* op_rope_kv_write: rotate q and k of qkv [B][(nq + 2 nkv) d] (fp32; q heads,
 * then k heads, then v heads) at positions[b] with the rotate-half pairing
 * (element i with i + d/2, angle p * theta^(-2i/d)), write rotated q to q_out
 * [B][nq][d] fp32, and store k / k_scale and v / v_scale, rounded to the cache
 * format (BF16 or e4m3), at block bt[b][p / 16], slot p % 16 of the pools
 * kpool, vpool [num_blocks + 1][nkv][16][d]. ("Kernels, Fusion & CUDA Graphs",
 * "Fix 1: kernel fusion": RoPE + KV-cache write.) */
int op_rope_kv_write(int B, const float* qkv, int nq, int nkv, int d, const int32_t* positions,
                     const int32_t* bt, int bt_stride, int max_pos, float theta, void* kpool,
                     void* vpool, int num_blocks, int kv_dtype, float k_scale, float v_scale,
                     float* q_out, uint32_t* err, void* stream);

/* op_paged_attention: out[b][h] = sum_t softmax_t(q[b][h] . K_t / sqrt(d)) V_t
 * over t < seq_lens[b], K_t and V_t (times k_scale, v_scale) gathered through
 * bt; query head h reads KV head h / (nq / nkv). q [B][nq][d] fp32; out
 * [B][nq * d] fp32. Split-K over the context with the launch geometry the
 * decode step uses for a table of bt_stride entries. ("GPU Inference
 * Internals", "The KV-Cache Ledger" and "Kernels: FlashAttention and the Memory
 * Hierarchy".) */
int op_paged_attention(int B, const float* q, int nq, int nkv, int d, const void* kpool,
                       const void* vpool, int kv_dtype, float k_scale, float v_scale,
                       const int32_t* bt, int bt_stride, const int32_t* seq_lens, int num_blocks,
                       float* out, uint32_t* err, void* stream);

/* Size in bytes of the device array op_paged_attention_noalloc works in. */
#define MBT_NOALLOC_SCRATCH_BYTES (8u << 20)

/* op_paged_attention_noalloc: op_paged_attention for callers that cannot
 * allocate device memory when they run attention -- processes that reserve
 * nearly all HBM for their KV pool up front (a new allocation would fail or
 * fragment it), latency-critical paths where cudaMalloc / cudaFree may
 * synchronise the device, runtimes that forbid allocation after start-up. The
 * paper has no counterpart; this is a property of the library, not of the
 * method.
 * Same arguments, result and launch geometry as op_paged_attention, but its
 * scratch (split partials, (max, sum) pairs, merge tickets) is a file-scope
 * device array of MBT_NOALLOC_SCRATCH_BYTES that every GPU loading the library
 * holds until the process exits; it calls no cudaMalloc, cudaFree or other
 * allocating routine. The scratch needed is about B * nq * splits * (4 d + 8)
 * bytes (splits as op_paged_attention chooses them); a call needing more than
 * the array returns MBT_ERR_SCRATCH before doing any work.
 * All calls share the array and it keeps the last call's contents (the
 * tickets are cleared at every call): calls that overlap on the GPU race, so
 * keep them in one stream order. The first call on a device also does the
 * set-up (looks up the array's device address with that device current); make
 * it before any stream capture. */
int op_paged_attention_noalloc(int B, const float* q, int nq, int nkv, int d, const void* kpool,
                               const void* vpool, int kv_dtype, float k_scale, float v_scale,
                               const int32_t* bt, int bt_stride, const int32_t* seq_lens,
                               int num_blocks, float* out, uint32_t* err, void* stream);

/* op_paged_attention_noalloc_limit: MBT_NOALLOC_SCRATCH_BYTES, as built. */
size_t op_paged_attention_noalloc_limit(void);

#ifdef __cplusplus
}
#endif
#endif /* MBT_OPS_H_ */
