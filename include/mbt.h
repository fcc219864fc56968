/*
 * mbt.h -- C ABI of the GB300 decode-step library (libmbt.so).
 *
 * One decode step of a dense Llama-style decoder on one GPU: per layer a fused
 * residual-add + RMSNorm, a fused QKV projection, RoPE fused with the paged
 * KV-cache write, split-K paged decode attention with grouped-query heads, the
 * O projection, a fused gate+up projection with the SiLU-multiply epilogue and
 * the down projection; then the final norm, the LM head and a fused greedy
 * arg-max. The step is replayed as one CUDA graph per captured batch size.
 *
 * Where each operation is defined (page title, section):
 *   - the per-layer operation list and the eager/graph step model:
 *     "CUDA graphs & kernel fusion", "Direct answer";
 *   - the fused kernels (QKV, gate+up, residual add + RMSNorm, SiLU x mul,
 *     RoPE + KV-cache write, attention, sampling): "Kernels, Fusion & CUDA
 *     Graphs", "Fix 1: kernel fusion" table;
 *   - graph capture per batch size, the ladder 1, 2, 4, then every 8, padding
 *     to the next captured size, static input buffers, eager fallback above the
 *     top size: "Kernels, Fusion & CUDA Graphs", "Fix 2: CUDA graphs", and
 *     "CUDA graphs & kernel fusion", "Deep dive";
 *   - paged KV cache, FP8 weights and KV, dequantisation fused into the matmul:
 *     "Kernel Fusion for Large-Scale LLM Inference", section 11;
 *   - KV bytes per token for grouped-query attention: "GPU Inference
 *     Internals", "The KV-Cache Ledger".
 *
 * Conventions for every entry point:
 *   - Return 0 (MBT_OK) on success or a negative MBT_ERR_* code. No exception
 *     or C++ object crosses the boundary. mbt_status_string() names a code.
 *   - "device" pointers are CUDA device memory of the current device; "host"
 *     pointers are ordinary host memory. `stream` is a cudaStream_t (NULL = the
 *     legacy default stream). Calls that take a stream are asynchronous on it.
 *   - Handles are not thread-safe: one host thread at a time per model.
 *   - Errors a kernel detects (an out-of-range token id, block id, position or
 *     seq_len, a non-finite logit) never trap: the kernel skips the access,
 *     sets a bit in the model's device error word and carries on. Read and
 *     clear the word with model_poll_errors().
 */
#ifndef MBT_H_
#define MBT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MBT_OK               0
#define MBT_ERR_BAD_ARG     (-1)   /* null pointer, bad size or stride, wrong handle pairing */
#define MBT_ERR_BATCH       (-2)   /* B <= 0 */
#define MBT_ERR_CUDA        (-3)   /* a CUDA runtime call failed */
#define MBT_ERR_OOM         (-4)   /* device allocation failed */
#define MBT_ERR_BLOB        (-5)   /* malformed weight/config blob */
#define MBT_ERR_UNSUPPORTED (-6)   /* shape the kernels do not support */
#define MBT_ERR_NO_DEVICE   (-7)   /* no CUDA device, or not sm_103 */
#define MBT_ERR_SCRATCH     (-8)   /* request larger than a fixed scratch area */

/* ---- device error word bits (model_poll_errors) ----------------------- */
#define MBT_DEV_TOKEN_RANGE   0x1u   /* token id < 0 or >= vocab (token 0 used)   */
#define MBT_DEV_BLOCK_RANGE   0x2u   /* block id < 0 or > num_blocks (write/read skipped) */
#define MBT_DEV_POS_RANGE     0x4u   /* position < 0 or >= max_pos (write skipped) */
#define MBT_DEV_SEQLEN_RANGE  0x8u   /* seq_len < 1 or beyond the block table (row output 0) */
#define MBT_DEV_NONFINITE     0x10u  /* NaN logit met by the arg-max                */
#define MBT_DEV_WAIT_LIMIT    0x20u  /* a tensor-core kernel's pipeline wait timed out (its output is skipped) */

/* ---- weight/config blob ------------------------------------------------ *
 * A blob is one byte buffer: an mbt_blob_header at offset 0, an array of
 * n_tensors mbt_blob_tensor entries at table_offset, and tensor data at the
 * offsets the entries give (each 256-byte aligned). Matrices are row-major
 * [rows][cols], one output channel per row. FP8 matrices are e4m3 codes with
 * one fp32 scale per row in a separate MBT_T_S_* tensor (value = e4m3 * scale).
 * Gains (g_*) and the embedding are always BF16.
 *   w_qkv rows: n_q_heads*head_dim query rows, then n_kv_heads*head_dim key
 *               rows, then n_kv_heads*head_dim value rows.
 *   w_gu rows:  ffn gate rows, then ffn up rows.                            */
#define MBT_BLOB_MAGIC   "MBTBLOB1"
#define MBT_BLOB_VERSION 1u
#define MBT_DTYPE_BF16   0u
#define MBT_DTYPE_E4M3   1u
#define MBT_DTYPE_F32    2u

enum mbt_tensor_kind {
  MBT_T_EMBED = 0, MBT_T_G_ATTN = 1, MBT_T_W_QKV = 2, MBT_T_S_QKV = 3,
  MBT_T_W_O = 4, MBT_T_S_O = 5, MBT_T_G_FFN = 6, MBT_T_W_GU = 7, MBT_T_S_GU = 8,
  MBT_T_W_DOWN = 9, MBT_T_S_DOWN = 10, MBT_T_G_FINAL = 11, MBT_T_LM_HEAD = 12,
  MBT_T_S_LM = 13
};

typedef struct mbt_blob_header {
  char     magic[8];        /* MBT_BLOB_MAGIC, not NUL-terminated           */
  uint32_t version;         /* MBT_BLOB_VERSION                               */
  uint32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  uint32_t weight_dtype;    /* MBT_DTYPE_BF16 or MBT_DTYPE_E4M3              */
  uint32_t kv_dtype;        /* MBT_DTYPE_BF16 or MBT_DTYPE_E4M3              */
  uint32_t block_size;      /* tokens per KV block; must be 16               */
  uint32_t max_pos;         /* positions 0..max_pos-1 are valid              */
  float    eps;             /* RMSNorm epsilon (inside the square root)       */
  float    rope_theta;      /* RoPE base                                      */
  uint32_t n_tensors;
  uint32_t reserved;
  uint64_t table_offset;    /* byte offset of the tensor table               */
} mbt_blob_header;          /* 80 bytes */

typedef struct mbt_blob_tensor {
  uint32_t kind;            /* enum mbt_tensor_kind                          */
  int32_t  layer;           /* 0..n_layers-1, or -1 for global tensors        */
  uint32_t dtype;           /* MBT_DTYPE_*                                    */
  uint32_t reserved;
  uint64_t rows, cols;      /* cols = 1 for vectors                           */
  uint64_t offset, bytes;   /* data location in the blob                      */
} mbt_blob_tensor;          /* 48 bytes */

typedef struct mbt_model mbt_model;
typedef struct mbt_kv mbt_kv;

/* model_create: parse and validate the blob (magic, version, dims, dtypes,
 * every tensor's presence, shape, offset and size), copy the weights into
 * device memory the library owns and build the RoPE cos/sin table.
 *   blob, bytes:    the blob; host memory, or device memory if blob_is_device.
 *                   The caller keeps ownership and may free it on return.
 *   stream:         stream for the copies; the call synchronises it.
 *   out:            receives the handle.
 * Supported shapes: head_dim 64 or 128; hidden, n_q_heads*head_dim and ffn
 * multiples of 16; n_q_heads a multiple of n_kv_heads; block_size 16.
 * Errors: MBT_ERR_BLOB, MBT_ERR_UNSUPPORTED, MBT_ERR_OOM, MBT_ERR_CUDA,
 * MBT_ERR_NO_DEVICE. */
int model_create(const void* blob, size_t bytes, int blob_is_device, void* stream,
                 mbt_model** out);

/* model_destroy: free the weights, workspaces and graphs. NULL is a no-op. */
int model_destroy(mbt_model* m);

/* model_info: copy the model's header (tensor table fields zeroed) to *out (host). */
int model_info(const mbt_model* m, mbt_blob_header* out);

/* kv_bytes: device bytes of a KV pool with num_blocks caller blocks (one
 * reserved null block is added). 0 if num_blocks < 1. */
size_t kv_bytes(const mbt_model* m, int num_blocks);

/* kv_alloc: create a paged KV cache. Layout in device memory (row-major):
 *   [layer][2 (K, V)][num_blocks + 1][n_kv_heads][16 tokens][head_dim]
 * in the model's KV dtype (BF16, or e4m3 storing value / scale). Block ids
 * 0..num_blocks-1 belong to the caller; id num_blocks is the null block that
 * padded batch rows write to. Token p of a sequence lives in block
 * table[p / 16] at slot p % 16.
 *   device_mem_or_null: caller memory of at least kv_bytes() bytes (the caller
 *                   keeps ownership and must outlive the handle), or NULL to
 *                   let the library allocate.
 * Per-layer K and V scales start at 1.0. Contents start uninitialised.
 * Errors: MBT_ERR_BAD_ARG (num_blocks < 1), MBT_ERR_OOM. */
int kv_alloc(mbt_model* m, int num_blocks, void* device_mem_or_null, mbt_kv** out);

/* kv_free: release the handle (and the pool if the library allocated it). */
int kv_free(mbt_kv* kv);

/* kv_pool: device address and size in bytes of the pool (layout above). */
int kv_pool(const mbt_kv* kv, void** pool, size_t* bytes);

/* kv_set_scales: per-layer fp32 dequantisation scales for an FP8 cache (host
 * arrays of n_layers entries each). A stored code c means e4m3(c) * scale.
 * Must be called before model_capture (graphs bake the scales in). */
int kv_set_scales(mbt_kv* kv, const float* k_scales, const float* v_scales);

/* model_capture: capture one CUDA graph per batch size in ladder[0..n) (sorted
 * ascending, each >= 1), bound to this kv, for block tables of up to
 * max_blocks_per_seq entries per row. ladder == NULL uses 1, 2, 4 and then
 * every 8 up to 64. Graphs replay on any stream. Capture runs every rung once
 * eagerly first (warm-up) on `stream` and synchronises it. After capture
 * decode_step pads a batch of B rows to the smallest captured size >= B and
 * replays its graph; B above the largest size, another kv, or a block table
 * wider than max_blocks_per_seq entries (bt_stride) runs eagerly. An eager
 * step never invalidates the graphs: when it needs more workspace than they
 * were captured with, it uses a separate one.
 * Errors: MBT_ERR_BAD_ARG, MBT_ERR_OOM, MBT_ERR_CUDA. */
int model_capture(mbt_model* m, mbt_kv* kv, const int* ladder, int n,
                  int max_blocks_per_seq, void* stream);

/* model_set_eager: 1 = never replay graphs (debug mode), 0 = use them. */
int model_set_eager(mbt_model* m, int eager);

/* decode_step: one decode step for B sequences. All array pointers are
 * caller-owned DEVICE memory:
 *   token_ids[B]      int32  token fed at this step
 *   positions[B]      int32  its position p (0-based); K and V are written to
 *                            block block_tables[b][p / 16], slot p % 16
 *   block_tables[B][bt_stride] int32 physical block ids of each sequence
 *   seq_lens[B]       int32  tokens attended over, the new one included
 *                            (normally positions[b] + 1); at most
 *                            bt_stride * 16: a row beyond its table is
 *                            flagged MBT_DEV_SEQLEN_RANGE and attends over
 *                            nothing, on the graph and the eager path alike
 *   next_ids[B]       int32  out: arg-max of the logits (lowest id on ties)
 *   logits_or_null    float  out: [B][vocab] fp32 logits, or NULL
 * Asynchronous on `stream`. Returns MBT_ERR_BATCH for B <= 0, MBT_ERR_BAD_ARG
 * for a null pointer, bt_stride < 1 or a kv of another model, MBT_ERR_CUDA if
 * a launch fails. Device-detected range errors go to the error word. */
int decode_step(mbt_model* m, mbt_kv* kv, int B, const int32_t* token_ids,
                const int32_t* positions, const int32_t* block_tables, int bt_stride,
                const int32_t* seq_lens, int32_t* next_ids, float* logits_or_null,
                void* stream);

/* Sampling parameters of decode_step_sample (host struct). */
#define MBT_TOPK_MAX 1024
typedef struct mbt_sampling {
  float    temperature;     /* > 0: the logits are divided by it              */
  int32_t  top_k;           /* 0 = no top-k cut, else 1..MBT_TOPK_MAX         */
  float    top_p;           /* (0, 1]; 1 = no top-p cut                       */
  uint32_t reserved;        /* 0                                              */
  uint64_t seed;            /* generator key                                  */
  uint64_t step;            /* generator counter word: a new value per step    */
} mbt_sampling;             /* 32 bytes */

/* decode_step_sample: decode_step with the next token drawn instead of taken
 * by arg-max ("Kernels, Fusion & CUDA Graphs", "Fix 1: kernel fusion", the
 * "Sampling" row: softmax, top-k / top-p, sample). Per row b: z = logits / T;
 * the top_k largest z (a tie at the boundary keeps the lower id); softmax
 * over them; the shortest prefix in order of decreasing probability whose
 * probabilities reach top_p; then the Gumbel-max draw over that prefix: the
 * token with the largest z + g, g = -log(-log(u)), u from Philox4x32-10 with
 * key (seed mod 2^32, seed div 2^32) and counter (token id, b, step mod 2^32,
 * step div 2^32), u = (floor(x / 512) + 1/2) / 2^23 of its first word x.
 * With top_k = 0 and top_p = 1 the draw runs inside the LM head's epilogue
 * and the logits never leave the chip; otherwise the LM head writes the
 * logits once (B x vocab fp32) and a per-row kernel selects, normalises and
 * draws. top_p < 1 with top_k = 0 applies top-p to the MBT_TOPK_MAX largest
 * logits. Always runs eagerly (graphs, if any, stay valid). Arguments and
 * errors as decode_step; MBT_ERR_BAD_ARG also for params out of range.
 * logits_or_null receives the raw (unscaled) logits. */
int decode_step_sample(mbt_model* m, mbt_kv* kv, int B, const int32_t* token_ids,
                       const int32_t* positions, const int32_t* block_tables, int bt_stride,
                       const int32_t* seq_lens, const mbt_sampling* params, int32_t* next_ids,
                       float* logits_or_null, void* stream);

/* prefill: ingest the prompt tokens[0..n) of one sequence, at positions
 * start_pos .. start_pos + n - 1, in passes of up to 128 tokens through the
 * whole layer stack ("GPU Inference Internals", "Roofline: Why Decode Is
 * Memory-Bound": prefill works on the whole prompt at once, 2 x params x n
 * FLOPs, compute-bound; "Kernel Fusion for Large-Scale LLM Inference",
 * section 12: time to first token). Each prompt token's K and V are written
 * where decode_step would write them (block block_table[p / 16], slot p % 16)
 * with the same rounding, each token attends causally over positions 0..p
 * (positions before start_pos must already be in the cache), and the arg-max
 * of the last token's logits goes to next_id. Projections run on the tensor
 * cores for passes of 16 tokens or more.
 *   tokens[n]            int32 device
 *   block_table[bt_len]  int32 device: the sequence's blocks; bt_len * 16 >= start_pos + n
 *   next_id[1]           int32 device, out
 *   logits_or_null       float device [vocab], out: the last token's logits, or NULL
 * Runs eagerly (no graph) and asynchronously on `stream`; captured graphs stay
 * valid. Errors: MBT_ERR_BATCH (n < 1), MBT_ERR_BAD_ARG (a null pointer,
 * start_pos < 0, start_pos + n beyond max_pos or beyond the table, a kv of
 * another model), MBT_ERR_OOM, MBT_ERR_CUDA. Device-detected range errors go
 * to the error word. */
int prefill(mbt_model* m, mbt_kv* kv, int n, const int32_t* tokens, int start_pos,
            const int32_t* block_table, int bt_len, int32_t* next_id, float* logits_or_null, void* stream);

/* model_poll_errors: synchronise `stream`, return the device error word in
 * *bits (host) and clear it. */
int model_poll_errors(mbt_model* m, void* stream, uint32_t* bits);

/* model_stats: kernels launched by one step at batch B (graph nodes when a
 * graph serves B, else the eager launch count), and whether a graph serves B. */
int model_stats(mbt_model* m, int B, int* kernels_per_step, int* uses_graph);

/* status_string: static text for a status code. */
const char* status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* MBT_H_ */
