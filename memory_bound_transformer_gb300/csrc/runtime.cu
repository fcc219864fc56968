// Decode-step executor and the C ABI (include/mbt.h).
//
// The executor issues the per-layer kernel sequence of one decode step
// ("CUDA graphs & kernel fusion", "Direct answer": norms, QKV/O projections,
// attention, gate/up/down, activations, residual adds, repeated per layer) and
// captures it as one CUDA graph per batch size of a ladder, padding the live
// batch to the next captured size ("Kernels, Fusion & CUDA Graphs", "Fix 2:
// CUDA graphs"; "CUDA graphs & kernel fusion", "Deep dive": warm-up before
// capture, static input buffers, eager fallback).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"

using namespace mbt;

namespace {

// GEMV work-queue counters per step (one per launch and K split)
constexpr int kSchedCap = 8192;
// Fewest rows that run on the tensor cores (below: the CUDA-core GEMV). The
// CUDA-core GEMV re-reads the weights for every 8 rows and keeps 8 rows x 32
// accumulators per thread at one CTA per SM; measured on the 8B-class BF16
// step (ms per step at 1 / 2 / 3 / 4 / 8 rows): CUDA cores 2.94 / 3.56 / 5.00
// / 5.16 / 9.07 against tensor cores - / 3.52 / 3.46 / 3.47 / 3.63, so every
// batch from 2 rows on runs on the tensor cores.
#ifndef MBT_TC_MIN_ROWS
#define MBT_TC_MIN_ROWS 2
#endif
constexpr int kTcMinRows = MBT_TC_MIN_ROWS;
// Prompt tokens per prefill pass (rows of one pass through the layers).
constexpr int kPrefillChunk = 128;



struct Layer {
  const void* w_qkv; const float* s_qkv;
  const void* w_o; const float* s_o;
  const void* w_gu; const float* s_gu;
  const void* w_down; const float* s_down;
  const bf16* g_attn; const bf16* g_ffn;
};

// Launch geometry of one step at R rows and block tables of `mbs` entries.
struct Plan {
  int R = 0, mbs = 0;
  int attn_bps = 0, attn_nsplit = 0;
  int ns_qkv = 1, ns_o = 1, ns_down = 1;   // split-K counts of the residual-feeding projections
  int g_lm = 1;                            // LM-head CTAs (arg-max partials per row)
  bool use_tc = false;                     // tensor-core GEMMs (batch 16..128, BF16 weights)
  int rp = 0;                              // rows padded to a multiple of 16 (tensor-core path)
  int kernels = 0;
};

// Sampling in place of the greedy arg-max (null: arg-max). mode 1: the draw
// is fused into the LM head's arg-max epilogue (temperature only, the logits
// stay on chip); mode 2: the LM head writes the logits to `z` (rows of vocab
// floats) and the top-k / top-p kernel draws from them.
struct SampleCfg {
  int mode; GumbelArgs gum; int k; float top_p; float* z;
};

// Device workspace for up to `cap` rows.
struct Workspace {
  int cap = 0, mbs_cap = 0;
  size_t part_o_elems = 0, part_ml_elems = 0;
  int ns_qkv_cap = 0, ns_delta_cap = 0, g_lm_cap = 0;
  void* mem = nullptr;
  float* r = nullptr; float* r2 = nullptr;           // residual ping-pong [cap][H]
  float* qkv = nullptr;                              // QKV partials [splits][cap][QKV]
  float* part_o = nullptr; float2* part_ml = nullptr; float* o = nullptr;
  float* delta = nullptr; float* delta2 = nullptr;   // O and down partials [splits][cap][H]
  float* act = nullptr; ArgmaxPart* lm_part = nullptr;
  int* attn_tickets = nullptr;
  int* sched = nullptr;                              // GEMV work-queue counters, zeroed each step
  int* tickets = nullptr; int tickets_cap = 0;       // tensor-core GEMM per-tile tickets (right after sched)
  float* ts_scratch = nullptr;                       // tensor-core GEMM partial sums
  int rp_cap = 0;                                    // tensor-core path: 16-bit high/low rows
  bf16* x_hl = nullptr; bf16* o_hl = nullptr; bf16* act_hl = nullptr;
  // e4m3 weights: the projections' inputs as e4m3 term rows [4][rp_cap][K]
  // (the norm output reuses x_hl's bytes) and their row scales
  uint8_t* o_t = nullptr; uint8_t* act_t = nullptr;
  float* x_s = nullptr; float* o_s = nullptr; float* act_s = nullptr;
  float* q = nullptr;                                // prefill: rotated queries [cap][nq * d]
  int* pf_tok = nullptr; int* pf_pos = nullptr; int* pf_sl = nullptr;   // prefill rows [cap]
  int* pf_bt = nullptr;                              // prefill block tables [cap][mbs_cap]
};

struct Graph {
  int R = 0;
  cudaGraphExec_t exec[2] = {nullptr, nullptr};   // [without logits, with logits]
  int nodes = 0;
};

}  // namespace

struct mbt_model {
  mbt_blob_header h;
  int device = 0, num_sms = 0;
  int wtype = W_BF16, kv8 = 0;
  StreamCfg stream;                 // L1 split and GEMV shared-memory budget of the batch 1..15 step
  void* wmem = nullptr;
  size_t wbytes = 0;
  const bf16* embed = nullptr; const bf16* g_final = nullptr;
  const void* lm = nullptr; const float* s_lm = nullptr;
  std::vector<Layer> layers;
  std::vector<TmaMap> wmaps;        // tensor maps of the BF16 weights: [layer][qkv, o, gu, down], lm head
  bool tc_ok = false;
  float2* rope = nullptr;
  uint32_t* err = nullptr;
  Workspace ws;                     // bound to the captured graphs (their kernels hold its addresses)
  Workspace ws_eager;               // eager steps the graph-bound workspace is too small for
  // graphs
  std::vector<Graph> graphs;
  mbt_kv* graph_kv = nullptr;
  int graph_mbs = 0;
  int eager = 0;
  void* statics = nullptr;
  int* s_tok = nullptr; int* s_pos = nullptr; int* s_sl = nullptr; int* s_bt = nullptr;
  int* s_next = nullptr; float* s_logits = nullptr;
  float* samp_z = nullptr; int samp_rows = 0;   // logits of a top-k / top-p step
};

struct mbt_kv {
  mbt_model* m = nullptr;
  int num_blocks = 0;
  void* pool = nullptr;
  size_t bytes = 0;
  bool owned = false;
  std::vector<float> k_scale, v_scale;
};

namespace {

#define MBT_CUDA(x)                                   \
  do {                                                \
    cudaError_t e_ = (x);                             \
    if (e_ != cudaSuccess) return MBT_ERR_CUDA;       \
  } while (0)

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t kv_layer_half_bytes(const mbt_model* m, int num_blocks) {
  const size_t esz = m->kv8 ? 1 : 2;
  return (size_t)(num_blocks + 1) * m->h.n_kv_heads * kBlockTokens * m->h.head_dim * esz;
}

Plan make_plan(const mbt_model* m, int R, int mbs) {
  Plan p;
  p.R = R;
  p.mbs = mbs;
  attn_plan(R, (int)m->h.n_kv_heads, mbs, m->num_sms,
            attn_ctas_per_sm(m->kv8, (int)(m->h.n_q_heads / m->h.n_kv_heads)), &p.attn_bps, &p.attn_nsplit);
  const int nb0 = std::min(R, 8);
  const int H = (int)m->h.hidden, Q = (int)(m->h.n_q_heads * m->h.head_dim), F = (int)m->h.ffn;
  const int L = (int)m->h.n_layers;
  p.use_tc = m->tc_ok && R >= kTcMinRows;
  if (p.use_tc) {
    // the stream-K GEMM leaves complete sums (no K-split partials) and runs
    // in launches of at most 64 rows
    p.rp = (R + 15) / 16 * 16;
    p.ns_qkv = p.ns_o = p.ns_down = 1;
    p.g_lm = ts_tiles(EPI_ARGMAX, (int)m->h.vocab);
    const int chunks = (R + kTsMaxRows - 1) / kTsMaxRows;
    // e4m3 weights: two term-split launches per layer (attention's and the SwiGLU's rows)
    p.kernels = 1 + (3 + 4 * chunks + (m->wtype == W_E4M3 ? 2 : 0)) * L + 2 + chunks;
    return p;
  }
  p.ns_qkv = 1;                                          // norm prologue: whole rows per CTA
  p.ns_o = gemv_plan(EPI_PARTIAL, m->wtype, nb0, H, Q, m->num_sms, 0, PRO_X, m->stream).nsplit;
  p.ns_down = gemv_plan(EPI_PARTIAL, m->wtype, nb0, H, F, m->num_sms, 0, PRO_X, m->stream).nsplit;
  const int mn = gemv_max_rows(EPI_ARGMAX, H, PRO_NORM);
  p.g_lm = gemv_plan(EPI_ARGMAX, m->wtype, std::min(nb0, mn), (int)m->h.vocab, H, m->num_sms, 0, PRO_NORM,
                     m->stream).grid;

  const int c8 = (R + 7) / 8;
  const int cn = (R + mn - 1) / mn;                      // chunks of the norm-prologue projections
  p.kernels = 1 + L * (2 * cn + 2 * c8 + 1) + cn + 1;
  return p;
}

void free_ws(Workspace& w) {
  if (w.mem) cudaFree(w.mem);
  w = Workspace();
}

// Capacities a workspace needs to serve R rows with block tables of mbs entries.
struct WsNeed {
  int cap, mbs_cap, ns_qkv, ns_delta, g_lm;
  size_t po, pml;
};

WsNeed ws_need(const mbt_model* m, const Workspace& w, int R, int mbs) {
  WsNeed n;
  n.cap = std::max(R, w.cap);
  n.mbs_cap = std::max(mbs, w.mbs_cap);
  n.ns_qkv = 1; n.ns_delta = 1; n.g_lm = 1;
  n.pml = 0;
  for (int r = 1; r <= n.cap; ++r) {
    Plan p = make_plan(m, r, n.mbs_cap);
    const int pairs = r * (int)m->h.n_kv_heads;
    // attn_plan never uses more splits than this, whatever the table width up to mbs_cap
    const int split_bound = std::max({1, (4 * m->num_sms + pairs - 1) / pairs, (n.mbs_cap + 511) / 512});
    n.pml = std::max(n.pml, (size_t)r * m->h.n_q_heads * split_bound);
    n.ns_qkv = std::max(n.ns_qkv, p.ns_qkv);
    n.ns_delta = std::max({n.ns_delta, p.ns_o, p.ns_down});
    n.g_lm = std::max(n.g_lm, p.g_lm);
  }
  n.po = n.pml * m->h.head_dim;
  return n;
}

bool ws_covers(const Workspace& w, const WsNeed& n) {
  return w.mem && n.cap <= w.cap && n.mbs_cap <= w.mbs_cap && n.po <= w.part_o_elems &&
         n.ns_qkv <= w.ns_qkv_cap && n.ns_delta <= w.ns_delta_cap && n.g_lm <= w.g_lm_cap;
}

// Grow workspace `w` to serve R rows with block tables of mbs entries. Growing
// the graph-bound workspace invalidates the captured graphs (they hold its old
// addresses), so callers grow it only while no graph exists (capture, or eager
// mode before any capture); eager steps beside live graphs use m->ws_eager.
int ensure_ws(mbt_model* m, Workspace& w, int R, int mbs) {
  const WsNeed n = ws_need(m, w, R, mbs);
  if (ws_covers(w, n)) return MBT_OK;
  if (cudaDeviceSynchronize() != cudaSuccess) return MBT_ERR_CUDA;
  if (&w == &m->ws) {
    for (auto& g : m->graphs)
      for (auto& e : g.exec) if (e) cudaGraphExecDestroy(e);
    m->graphs.clear();
    m->graph_kv = nullptr;
  }
  free_ws(w);
  const int cap = n.cap, mbs_cap = n.mbs_cap, ns_qkv = n.ns_qkv, ns_delta = n.ns_delta, g_lm = n.g_lm;
  const size_t po = n.po, pml = n.pml;
  const size_t H = m->h.hidden, Q = (size_t)m->h.n_q_heads * m->h.head_dim, F = m->h.ffn;
  const size_t QKV = (size_t)(m->h.n_q_heads + 2 * m->h.n_kv_heads) * m->h.head_dim;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off += align256(bytes); return o; };
  const size_t o_r = take((size_t)cap * H * 4), o_r2 = take((size_t)cap * H * 4);
  const size_t o_qkv = take((size_t)ns_qkv * cap * QKV * 4);
  const size_t o_po = take(po * 4), o_pml = take(pml * 8), o_o = take((size_t)cap * Q * 4);
  const size_t o_d = take((size_t)ns_delta * cap * H * 4), o_d2 = take((size_t)ns_delta * cap * H * 4);
  const size_t o_a = take((size_t)cap * F * 4);
  const size_t o_lp = take((size_t)g_lm * cap * sizeof(ArgmaxPart));
  const size_t o_tk = take((size_t)cap * m->h.n_kv_heads * 4);
  const int QKVn = (int)QKV, Hn = (int)H, Fn = (int)F, Vn = (int)m->h.vocab;
  const int tcap = std::max({ts_tiles(EPI_PARTIAL, QKVn), ts_tiles(EPI_PARTIAL, Hn), ts_tiles(EPI_SWIGLU, Fn),
                             ts_tiles(EPI_ARGMAX, Vn)});
  const size_t o_sc = take((size_t)(kSchedCap + tcap) * 4);
  const size_t o_ts = take(ts_scratch_floats(m->num_sms) * 4);
  const int rp_cap = (cap + 15) / 16 * 16;
  const size_t b_xhl = (size_t)2 * rp_cap * H * 2, b_ohl = (size_t)2 * rp_cap * Q * 2;
  const size_t b_ahl = (size_t)2 * rp_cap * F * 2;
  const size_t o_xhl = take(b_xhl), o_ohl = take(b_ohl), o_ahl = take(b_ahl);
  const bool t8 = m->wtype == W_E4M3;
  const size_t o_ot = take(t8 ? (size_t)kTerms * rp_cap * Q : 0), o_at = take(t8 ? (size_t)kTerms * rp_cap * F : 0);
  const size_t o_xs = take(t8 ? (size_t)3 * rp_cap * 4 : 0);
  const size_t o_q = take((size_t)cap * Q * 4);
  const size_t o_pf = take((size_t)cap * 3 * 4), o_pfbt = take((size_t)cap * mbs_cap * 4);
  void* mem = nullptr;
  if (cudaMalloc(&mem, off) != cudaSuccess) { cudaGetLastError(); return MBT_ERR_OOM; }
  char* base = (char*)mem;
  w.mem = mem; w.cap = cap; w.mbs_cap = mbs_cap;
  w.part_o_elems = po; w.part_ml_elems = pml;
  w.ns_qkv_cap = ns_qkv; w.ns_delta_cap = ns_delta; w.g_lm_cap = g_lm;
  w.r = (float*)(base + o_r); w.r2 = (float*)(base + o_r2); w.qkv = (float*)(base + o_qkv);
  w.part_o = (float*)(base + o_po); w.part_ml = (float2*)(base + o_pml);
  w.o = (float*)(base + o_o); w.delta = (float*)(base + o_d); w.delta2 = (float*)(base + o_d2);
  w.act = (float*)(base + o_a);
  w.lm_part = (ArgmaxPart*)(base + o_lp);
  w.attn_tickets = (int*)(base + o_tk);
  w.sched = (int*)(base + o_sc);
  w.tickets = w.sched + kSchedCap; w.tickets_cap = tcap;
  w.ts_scratch = (float*)(base + o_ts);
  w.rp_cap = rp_cap;
  w.x_hl = (bf16*)(base + o_xhl); w.o_hl = (bf16*)(base + o_ohl); w.act_hl = (bf16*)(base + o_ahl);
  if (t8) {
    w.o_t = (uint8_t*)(base + o_ot); w.act_t = (uint8_t*)(base + o_at);
    w.x_s = (float*)(base + o_xs); w.o_s = w.x_s + rp_cap; w.act_s = w.o_s + rp_cap;
  }
  w.q = (float*)(base + o_q);
  w.pf_tok = (int*)(base + o_pf); w.pf_pos = w.pf_tok + cap; w.pf_sl = w.pf_pos + cap;
  w.pf_bt = (int*)(base + o_pfbt);
  // attention tickets start at zero and every launch leaves them at zero; the
  // high/low activation rows start at zero so padding rows never hold NaN bits
  if (cudaMemset(mem, 0, off) != cudaSuccess) return MBT_ERR_CUDA;
  return MBT_OK;
}

// Inputs of a norm-prologue projection: x = rmsnorm(r_in + sum of n_delta
// partials) * gamma, new residual to r_out.
struct NormIn {
  const float* r_in; const float* delta; int n_delta; const bf16* gamma; float* r_out;
};

// One GEMV over R rows, issued in chunks of at most 8 rows (fewer when the
// fp32 x tile of an unsplittable launch would not fit in shared memory).
cudaError_t gemv_rows(const mbt_model* m, const Workspace& ws, int epi, const NormIn* nin, const void* W, const float* sc,
                      int N, int K, const float* x, int R, int nsplit, int grid_fixed, float* out,
                      long long split_stride, int ldo, float* act, int lda, float* logits,
                      ArgmaxPart* part, int part_ld, cudaStream_t s, uint32_t prefetch = 0,
                      int* sched_used = nullptr, const GumbelArgs* gum = nullptr) {
  const int pro = nin ? PRO_NORM : PRO_X;
  const int step = gemv_max_rows(epi, K, pro);
  for (int b0 = 0; b0 < R; b0 += step) {
    const int nb = std::min(step, R - b0);
    GemvLaunch g = gemv_plan(epi, m->wtype, nb, N, K, m->num_sms, epi == EPI_PARTIAL ? nsplit : 0, pro, m->stream);
    if (grid_fixed > 0) g.grid = grid_fixed;
    GemvArgs a;
    memset(&a, 0, sizeof(a));
    a.W = W; a.scale = sc; a.wtype = m->wtype; a.N = N; a.K = K;
    a.x = x ? x + (size_t)b0 * K : nullptr; a.ldx = K; a.nb = nb;
    if (nin) {
      a.r_in = nin->r_in + (size_t)b0 * K;
      a.delta = nin->delta ? nin->delta + (size_t)b0 * K : nullptr;
      a.n_delta = nin->n_delta; a.delta_stride = (long long)R * K;
      a.gamma = nin->gamma; a.eps = m->h.eps;
      a.r_out = nin->r_out + (size_t)b0 * K;
    }
    a.out = out ? out + (size_t)b0 * ldo : nullptr; a.split_stride = split_stride; a.ldo = ldo;
    a.act = act ? act + (size_t)b0 * lda : nullptr; a.lda = lda;
    a.logits = logits ? logits + (size_t)b0 * m->h.vocab : nullptr; a.ldl = (int)m->h.vocab;
    a.part = part ? part + b0 : nullptr; a.part_ld = part_ld;
    a.err = m->err;
    a.prefetch_bytes = prefetch;
    if (gum) { a.gum = *gum; a.gum.row0 = b0; }
    // work-queue tail: a fixed share of each CTA's rows, the rest claimed one
    // group at a time (kernels that prefetch their whole slice keep it fixed)
    const int sg = gemv_queue_static_groups(g, N);
    if (sched_used && prefetch != 0xffffffffu && sg >= 0 && *sched_used + g.nsplit <= kSchedCap) {
      a.sched = ws.sched + *sched_used;
      a.static_groups = sg;
      *sched_used += g.nsplit;
    }
    cudaError_t e = gemv_launch(epi, pro, a, g, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Prefill form of the attention step: the chunk's rows are consecutive
// tokens of one sequence, so every row's K and V must be in the cache before
// any row attends (row i reads rows < i of the same chunk). RoPE + KV write
// runs as its own kernel over all rows (queries rotated into w.q), then the
// attention kernel reads the queries and the cache, writing nothing; it is an
// ordinary launch, so its early cache reads see the writes just made.
cudaError_t prefill_rope_kv(const mbt_model* m, const Workspace& w, const mbt_kv* kv, int l, int R, int ns_qkv,
                            const int* pos, const int* bt, int bt_stride, cudaStream_t s) {
  const int d = (int)m->h.head_dim, nq = (int)m->h.n_q_heads, nkv = (int)m->h.n_kv_heads;
  const int QKV = (nq + 2 * nkv) * d;
  const size_t half = kv_layer_half_bytes(m, kv->num_blocks);
  char* kbase = (char*)kv->pool + 2 * half * (size_t)l;
  RopeKvArgs rk = {};
  rk.B = R; rk.qkv = w.qkv; rk.nsplit = ns_qkv; rk.split_stride = (long long)R * QKV; rk.ld_qkv = QKV;
  rk.nq = nq; rk.nkv = nkv; rk.d = d; rk.positions = pos; rk.bt = bt; rk.bt_stride = bt_stride;
  rk.max_pos = (int)m->h.max_pos; rk.rope = m->rope; rk.q_out = w.q;
  rk.kpool = kbase; rk.vpool = kbase + half; rk.num_blocks = kv->num_blocks;
  rk.kv_fp8 = m->kv8; rk.k_scale = kv->k_scale[l]; rk.v_scale = kv->v_scale[l]; rk.err = m->err;
  return launch_rope_kv_write(rk, s);
}

// After an LM head that wrote the logits to smp->z: the top-k / top-p draw.
cudaError_t sample_from_logits(const mbt_model* m, const SampleCfg* smp, int R, int* next_ids, cudaStream_t s) {
  TopKArgs t = {};
  t.B = R; t.V = (int)m->h.vocab; t.ldl = (int)m->h.vocab; t.logits = smp->z; t.inv_t = smp->gum.inv_t;
  t.k = smp->k; t.top_p = smp->top_p; t.gum = smp->gum; t.next_ids = next_ids; t.err = m->err;
  return launch_sample_topk(t, s);
}

// Prefill tail: final norm and LM head for the chunk's last row only (the
// sequence's next token); the residual of that row plus the down projection's
// pending partials, normalised into w.r2, then the arg-max GEMV.
int lm_head_last_row(mbt_model* m, const Workspace& w, const Plan& p, int* next_ids, float* logits, cudaStream_t s) {
  const int R = p.R, H = (int)m->h.hidden, V = (int)m->h.vocab;
  const size_t last = (size_t)(R - 1) * H;
  AddNormArgs an{1, H, w.r + last, w.delta2 + last, p.ns_down, (long long)R * H, m->g_final, m->h.eps, w.r2,
                 nullptr, 0, 0};
  MBT_CUDA(launch_add_rmsnorm(an, s));
  const GemvLaunch g = gemv_plan(EPI_ARGMAX, m->wtype, 1, V, H, m->num_sms, 0, PRO_X, m->stream);
  if (g.grid > w.g_lm_cap * w.cap) return MBT_ERR_UNSUPPORTED;
  MBT_CUDA(gemv_rows(m, w, EPI_ARGMAX, nullptr, m->lm, m->s_lm, V, H, w.r2, 1, 1, g.grid, nullptr, 0, 0,
                     nullptr, 0, logits, w.lm_part, 1, s));
  MBT_CUDA(launch_argmax_reduce(1, w.lm_part, 1, g.grid, next_ids, m->err, s));
  return MBT_OK;
}

// Layers, final norm and LM head at batch 16..128 on the tensor cores: each
// projection reads BF16 high/low activation rows written by its producer
// (residual add + RMSNorm, attention, the gate/up GEMM's SwiGLU epilogue).
int run_layers_tc(mbt_model* m, const Workspace& w, mbt_kv* kv, const Plan& p, const int* pos, const int* bt, int bt_stride,
                  const int* sl, int* next_ids, float* logits, cudaStream_t s, bool prefill,
                  const SampleCfg* smp) {
  const int R = p.R, Rp = p.rp;
  const int H = (int)m->h.hidden, d = (int)m->h.head_dim;
  const int nq = (int)m->h.n_q_heads, nkv = (int)m->h.n_kv_heads;
  const int Q = nq * d, F = (int)m->h.ffn, V = (int)m->h.vocab;
  const int QKV = (nq + 2 * nkv) * d;
  const size_t half = kv_layer_half_bytes(m, kv->num_blocks);
  const long long rh = (long long)R * H;
  // e4m3 weights: the projections read e4m3 term rows (the 16-bit rows that
  // attention and the SwiGLU epilogue write are FP16 and are split into terms);
  // BF16 weights: BF16 high/low rows
  const int f16 = m->wtype == W_E4M3;
  uint8_t* x_t = reinterpret_cast<uint8_t*>(w.x_hl);
  // one projection over the R rows, in launches of at most 64 rows that read
  // the activation rows from their first row on
  auto gemm = [&](int epi, const TmaMap& wm, const void* xbuf, const float* xs, int K,
                  const TcArgs& base) -> cudaError_t {
    for (int r0 = 0; r0 < R; r0 += kTsMaxRows) {
      const int rl = std::min(kTsMaxRows, R - r0), rc = (rl + 15) / 16 * 16;
      TmaMap xm;
      cudaError_t e = f16 ? tc_make_map_u8(&xm, xbuf, kTerms * Rp, K, rc) : tc_make_map(&xm, xbuf, 2 * Rp, K, rc);
      if (e != cudaSuccess) return e;
      TcArgs a = base;
      a.x_scale = xs;
      a.R = rl; a.Rp = rc; a.row0 = r0; a.rp_all = Rp;
      a.ts_scratch = w.ts_scratch; a.ts_tickets = w.tickets; a.tickets_cap = w.tickets_cap;
      e = ts_launch(m->wtype, epi, &wm, &xm, a, m->num_sms, s);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  };
  auto norm = [&](const float* delta, int n_delta, const bf16* gamma) {
    AddNormArgs an{R, H, w.r, delta, n_delta, rh, gamma, m->h.eps, nullptr, f16 ? nullptr : w.x_hl, Rp, 0};
    if (f16) { an.y_t = x_t; an.y_s = w.x_s; }
    return launch_add_rmsnorm(an, s);
  };
  auto partial = [&](const TmaMap& wm, const void* xbuf, const float* xs, const float* sc, int N, int K,
                     float* out) {
    TcArgs a = {};
    a.N = N; a.K = K; a.scale = sc;
    a.out = out; a.split_stride = (long long)R * N; a.ldo = N; a.err = m->err;
    return gemm(EPI_PARTIAL, wm, xbuf, xs, K, a);
  };
  const void* x_in = f16 ? (const void*)x_t : (const void*)w.x_hl;
  for (int l = 0; l < (int)m->h.n_layers; ++l) {
    const Layer& L = m->layers[l];
    const TmaMap* wm = &m->wmaps[(size_t)l * 4];
    char* kbase = (char*)kv->pool + 2 * half * (size_t)l;
    MBT_CUDA(norm(l ? w.delta2 : nullptr, l ? p.ns_down : 0, L.g_attn));
    MBT_CUDA(partial(wm[0], x_in, w.x_s, L.s_qkv, QKV, H, w.qkv));
    AttnArgs at = {};
    at.B = R; at.nq = nq; at.nkv = nkv; at.d = d;
    at.qkv = w.qkv; at.qkv_nsplit = p.ns_qkv; at.qkv_split_stride = (long long)R * QKV; at.ld_qkv = QKV;
    at.positions = pos; at.rope = m->rope; at.max_pos = (int)m->h.max_pos;
    at.kpool = kbase; at.vpool = kbase + half; at.kv_fp8 = m->kv8;
    at.k_scale = kv->k_scale[l]; at.v_scale = kv->v_scale[l];
    at.bt = bt; at.bt_stride = bt_stride; at.seq_lens = sl; at.num_blocks = kv->num_blocks;
    at.bps = p.attn_bps; at.nsplit = p.attn_nsplit;
    at.part_o = w.part_o; at.part_ml = w.part_ml; at.out = nullptr; at.tickets = w.attn_tickets; at.err = m->err;
    at.out_hl = w.o_hl; at.rp_hl = Rp; at.hl_f16 = f16;
    if (prefill) {
      MBT_CUDA(prefill_rope_kv(m, w, kv, l, R, p.ns_qkv, pos, bt, bt_stride, s));
      at.qkv = nullptr; at.q = w.q; at.no_pdl = 1;
    }
    MBT_CUDA(launch_attention(at, s));
    if (f16) MBT_CUDA(tc_to_terms(nullptr, w.o_hl, 1, R, Rp, Q, w.o_t, w.o_s, s));
    MBT_CUDA(partial(wm[1], f16 ? (const void*)w.o_t : (const void*)w.o_hl, w.o_s, L.s_o, H, Q, w.delta));
    MBT_CUDA(norm(w.delta, p.ns_o, L.g_ffn));
    TcArgs g = {};
    g.N = F; g.K = H; g.scale = L.s_gu; g.act_hl = w.act_hl; g.ld_act = F; g.err = m->err;
    g.hl_f16 = f16;
    MBT_CUDA(gemm(EPI_SWIGLU, wm[2], x_in, w.x_s, H, g));
    if (f16) MBT_CUDA(tc_to_terms(nullptr, w.act_hl, 1, R, Rp, F, w.act_t, w.act_s, s));
    MBT_CUDA(partial(wm[3], f16 ? (const void*)w.act_t : (const void*)w.act_hl, w.act_s, L.s_down, H, F, w.delta2));
  }
  if (prefill) return next_ids ? lm_head_last_row(m, w, p, next_ids, logits, s) : MBT_OK;
  MBT_CUDA(norm(w.delta2, p.ns_down, m->g_final));
  TcArgs a = {};
  a.N = V; a.K = H; a.scale = m->s_lm; a.logits = logits; a.ldl = V;
  a.part = w.lm_part; a.part_ld = R; a.err = m->err;
  if (smp && smp->mode == 1) a.gum = smp->gum;
  if (smp && smp->mode == 2) a.logits = smp->z;
  MBT_CUDA(gemm(EPI_ARGMAX, m->wmaps[(size_t)m->h.n_layers * 4], x_in, w.x_s, H, a));
  if (smp && smp->mode == 2) {
    MBT_CUDA(sample_from_logits(m, smp, R, next_ids, s));
    if (logits) MBT_CUDA(cudaMemcpyAsync(logits, smp->z, (size_t)R * V * 4, cudaMemcpyDeviceToDevice, s));
    return MBT_OK;
  }
  MBT_CUDA(launch_argmax_reduce(R, w.lm_part, R, p.g_lm, next_ids, m->err, s));
  return MBT_OK;
}

// The decode step over R rows whose inputs are already in device memory.
// Per layer: QKV projection with the RMSNorm prologue, attention with RoPE +
// KV write fused in, O projection, gate/up projection with the RMSNorm
// prologue and SwiGLU epilogue, down projection. The residual lives in two
// fp32 buffers (read one, write the other); projections with residual
// outputs leave split-K partials that the next norm prologue adds.
// With `prefill` the rows are consecutive prompt tokens of one sequence: the
// KV write is its own kernel before attention, and only the last row goes
// through the final norm and the LM head (none when next_ids is null).
int run_step(mbt_model* m, const Workspace& w, mbt_kv* kv, const Plan& p, const int* tok, const int* pos,
             const int* bt, int bt_stride, const int* sl, int* next_ids, float* logits,
             cudaStream_t s, bool prefill = false, const SampleCfg* smp = nullptr) {
  const int R = p.R;
  const int H = (int)m->h.hidden, d = (int)m->h.head_dim;
  const int nq = (int)m->h.n_q_heads, nkv = (int)m->h.n_kv_heads;
  const int Q = nq * d, F = (int)m->h.ffn, V = (int)m->h.vocab;
  const int QKV = (nq + 2 * nkv) * d;
  const size_t half = kv_layer_half_bytes(m, kv->num_blocks);
  const long long rh = (long long)R * H;

  EmbedNormArgs en{R, H, V, tok, m->embed, w.r, m->layers[0].g_attn, m->h.eps, nullptr, m->err,
                   w.sched, kSchedCap + w.tickets_cap, p.use_tc ? 0 : m->stream.carveout};
  MBT_CUDA(launch_embed_rmsnorm(en, s));
  if (p.use_tc) return run_layers_tc(m, w, kv, p, pos, bt, bt_stride, sl, next_ids, logits, s, prefill, smp);
  int sq = 0;                                        // work-queue counters taken so far
  for (int l = 0; l < (int)m->h.n_layers; ++l) {
    const Layer& L = m->layers[l];
    char* kbase = (char*)kv->pool + 2 * half * (size_t)l;
    // RMSNorm prologue + fused QKV projection
    NormIn n1{w.r, l ? w.delta2 : nullptr, l ? p.ns_down : 0, L.g_attn, w.r2};
    MBT_CUDA(gemv_rows(m, w, EPI_PARTIAL, &n1, L.w_qkv, L.s_qkv, QKV, H, nullptr, R, 1, 0, w.qkv,
                       (long long)R * QKV, QKV, nullptr, 0, nullptr, nullptr, 0, s, 0, &sq));
    // RoPE + paged KV write + split-K attention + merge
    AttnArgs at = {};
    at.B = R; at.q = nullptr; at.nq = nq; at.nkv = nkv; at.d = d;
    at.qkv = w.qkv; at.qkv_nsplit = 1; at.qkv_split_stride = (long long)R * QKV; at.ld_qkv = QKV;
    at.positions = pos; at.rope = m->rope; at.max_pos = (int)m->h.max_pos;
    at.kpool = kbase; at.vpool = kbase + half; at.kv_fp8 = m->kv8;
    at.k_scale = kv->k_scale[l]; at.v_scale = kv->v_scale[l];
    at.bt = bt; at.bt_stride = bt_stride; at.seq_lens = sl; at.num_blocks = kv->num_blocks;
    at.bps = p.attn_bps; at.nsplit = p.attn_nsplit;
    at.part_o = w.part_o; at.part_ml = w.part_ml; at.out = w.o; at.tickets = w.attn_tickets; at.err = m->err;
    at.carveout = m->stream.carveout;
    if (prefill) {
      MBT_CUDA(prefill_rope_kv(m, w, kv, l, R, 1, pos, bt, bt_stride, s));
      at.qkv = nullptr; at.q = w.q; at.no_pdl = 1;
    }
    MBT_CUDA(launch_attention(at, s));
    // O projection (residual partials); it starts during attention, whose
    // batch-1 form leaves HBM idle, so it prefetches all of its weights and
    MBT_CUDA(gemv_rows(m, w, EPI_PARTIAL, nullptr, L.w_o, L.s_o, H, Q, w.o, R, p.ns_o, 0, w.delta,
                       rh, H, nullptr, 0, nullptr, nullptr, 0, s, 0xffffffffu));
    // RMSNorm prologue + gate/up projection + SwiGLU epilogue
    NormIn n2{w.r2, w.delta, p.ns_o, L.g_ffn, w.r};
    MBT_CUDA(gemv_rows(m, w, EPI_SWIGLU, &n2, L.w_gu, L.s_gu, F, H, nullptr, R, 1, 0, nullptr, 0, 0,
                       w.act, F, nullptr, nullptr, 0, s, 0, &sq));
    // down projection (residual partials)
    MBT_CUDA(gemv_rows(m, w, EPI_PARTIAL, nullptr, L.w_down, L.s_down, H, F, w.act, R, p.ns_down, 0,
                       w.delta2, rh, H, nullptr, 0, nullptr, nullptr, 0, s, 0, &sq));
  }
  if (prefill) return next_ids ? lm_head_last_row(m, w, p, next_ids, logits, s) : MBT_OK;
  // final RMSNorm prologue + LM head with the arg-max epilogue, then the
  // cross-CTA reduction
  NormIn nf{w.r, w.delta2, p.ns_down, m->g_final, w.r2};
  float* lg = smp && smp->mode == 2 ? smp->z : logits;
  MBT_CUDA(gemv_rows(m, w, EPI_ARGMAX, &nf, m->lm, m->s_lm, V, H, nullptr, R, 1, p.g_lm, nullptr, 0, 0,
                     nullptr, 0, lg, w.lm_part, R, s, 0, &sq, smp && smp->mode == 1 ? &smp->gum : nullptr));
  if (smp && smp->mode == 2) {
    MBT_CUDA(sample_from_logits(m, smp, R, next_ids, s));
    if (logits) MBT_CUDA(cudaMemcpyAsync(logits, smp->z, (size_t)R * V * 4, cudaMemcpyDeviceToDevice, s));
    return MBT_OK;
  }
  MBT_CUDA(launch_argmax_reduce(R, w.lm_part, R, p.g_lm, next_ids, m->err, s, m->stream.carveout));
  return MBT_OK;
}

int find_tensor(const mbt_blob_tensor* t, uint32_t n, uint32_t kind, int layer) {
  for (uint32_t i = 0; i < n; ++i)
    if (t[i].kind == kind && t[i].layer == layer) return (int)i;
  return -1;
}

void destroy_graphs(mbt_model* m) {
  for (auto& g : m->graphs)
    for (auto& e : g.exec) if (e) cudaGraphExecDestroy(e);
  m->graphs.clear();
  m->graph_kv = nullptr;
  if (m->statics) cudaFree(m->statics);
  m->statics = nullptr;
}

}  // namespace

// ===========================================================================
// C ABI

extern "C" {

const char* status_string(int code) {
  switch (code) {
    case MBT_OK: return "ok";
    case MBT_ERR_BAD_ARG: return "bad argument";
    case MBT_ERR_BATCH: return "batch size must be >= 1";
    case MBT_ERR_CUDA: return "CUDA error";
    case MBT_ERR_OOM: return "out of device memory";
    case MBT_ERR_BLOB: return "malformed weight/config blob";
    case MBT_ERR_UNSUPPORTED: return "unsupported model shape";
    case MBT_ERR_NO_DEVICE: return "no usable CUDA device";
    case MBT_ERR_SCRATCH: return "request exceeds the fixed scratch area";
    default: return "unknown status";
  }
}

int model_create(const void* blob, size_t bytes, int blob_is_device, void* stream, mbt_model** out) {
  if (!blob || !out || bytes < sizeof(mbt_blob_header)) return MBT_ERR_BAD_ARG;
  *out = nullptr;
  cudaStream_t s = (cudaStream_t)stream;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return MBT_ERR_NO_DEVICE; }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MBT_ERR_NO_DEVICE;
  if (prop.major != 10 || prop.minor != 3) return MBT_ERR_NO_DEVICE;

  // header and table to host
  mbt_blob_header h;
  std::vector<unsigned char> hostcopy;
  const unsigned char* hb = nullptr;
  if (blob_is_device) {
    if (cudaMemcpy(&h, blob, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MBT_ERR_CUDA;
  } else {
    memcpy(&h, blob, sizeof(h));
    hb = (const unsigned char*)blob;
  }
  if (memcmp(h.magic, MBT_BLOB_MAGIC, 8) != 0 || h.version != MBT_BLOB_VERSION) return MBT_ERR_BLOB;
  if (h.n_layers < 1 || h.hidden < 16 || h.n_q_heads < 1 || h.n_kv_heads < 1 || h.ffn < 16 ||
      h.vocab < 1 || h.max_pos < 1 || h.n_tensors == 0 || h.n_tensors > 100000)
    return MBT_ERR_BLOB;
  if (!(h.eps > 0.f) || !(h.rope_theta > 1.f)) return MBT_ERR_BLOB;
  if (h.weight_dtype > 1 || h.kv_dtype > 1) return MBT_ERR_BLOB;
  if (h.block_size != (uint32_t)kBlockTokens) return MBT_ERR_UNSUPPORTED;
  if (h.head_dim != 64 && h.head_dim != 128) return MBT_ERR_UNSUPPORTED;
  if (h.n_q_heads % h.n_kv_heads != 0 || h.n_q_heads / h.n_kv_heads > 16) return MBT_ERR_UNSUPPORTED;
  if (h.hidden % 16 || (h.n_q_heads * h.head_dim) % 16 || h.ffn % 16) return MBT_ERR_UNSUPPORTED;
  if (h.hidden > 65536 || h.ffn > 262144 || h.vocab > (1u << 30)) return MBT_ERR_UNSUPPORTED;
  const size_t table_bytes = (size_t)h.n_tensors * sizeof(mbt_blob_tensor);
  if (h.table_offset > bytes || table_bytes > bytes - h.table_offset) return MBT_ERR_BLOB;
  std::vector<mbt_blob_tensor> tab(h.n_tensors);
  if (blob_is_device) {
    if (cudaMemcpy(tab.data(), (const char*)blob + h.table_offset, table_bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
      return MBT_ERR_CUDA;
  } else {
    memcpy(tab.data(), hb + h.table_offset, table_bytes);
  }

  // expected tensors: (kind, layer, dtype, rows, cols)
  struct Want { uint32_t kind; int layer; uint32_t dtype; uint64_t rows, cols; };
  std::vector<Want> want;
  const uint64_t H = h.hidden, Qd = (uint64_t)h.n_q_heads * h.head_dim, F = h.ffn, V = h.vocab;
  const uint64_t QKV = (uint64_t)(h.n_q_heads + 2 * h.n_kv_heads) * h.head_dim;
  const bool fp8 = h.weight_dtype == MBT_DTYPE_E4M3;
  const uint32_t wdt = fp8 ? MBT_DTYPE_E4M3 : MBT_DTYPE_BF16;
  want.push_back({MBT_T_EMBED, -1, MBT_DTYPE_BF16, V, H});
  for (int l = 0; l < (int)h.n_layers; ++l) {
    want.push_back({MBT_T_G_ATTN, l, MBT_DTYPE_BF16, H, 1});
    want.push_back({MBT_T_W_QKV, l, wdt, QKV, H});
    want.push_back({MBT_T_W_O, l, wdt, H, Qd});
    want.push_back({MBT_T_G_FFN, l, MBT_DTYPE_BF16, H, 1});
    want.push_back({MBT_T_W_GU, l, wdt, 2 * F, H});
    want.push_back({MBT_T_W_DOWN, l, wdt, H, F});
    if (fp8) {
      want.push_back({MBT_T_S_QKV, l, MBT_DTYPE_F32, QKV, 1});
      want.push_back({MBT_T_S_O, l, MBT_DTYPE_F32, H, 1});
      want.push_back({MBT_T_S_GU, l, MBT_DTYPE_F32, 2 * F, 1});
      want.push_back({MBT_T_S_DOWN, l, MBT_DTYPE_F32, H, 1});
    }
  }
  want.push_back({MBT_T_G_FINAL, -1, MBT_DTYPE_BF16, H, 1});
  want.push_back({MBT_T_LM_HEAD, -1, wdt, V, H});
  if (fp8) want.push_back({MBT_T_S_LM, -1, MBT_DTYPE_F32, V, 1});

  std::vector<int> idx(want.size());
  std::vector<size_t> dst(want.size());
  size_t total = 0;
  for (size_t i = 0; i < want.size(); ++i) {
    const Want& w = want[i];
    const int j = find_tensor(tab.data(), h.n_tensors, w.kind, w.layer);
    if (j < 0) return MBT_ERR_BLOB;
    const mbt_blob_tensor& t = tab[j];
    const uint64_t esz = w.dtype == MBT_DTYPE_BF16 ? 2 : w.dtype == MBT_DTYPE_E4M3 ? 1 : 4;
    if (t.dtype != w.dtype || t.rows != w.rows || t.cols != w.cols || t.bytes != w.rows * w.cols * esz)
      return MBT_ERR_BLOB;
    if (t.offset % 16 || t.offset > bytes || t.bytes > bytes - t.offset) return MBT_ERR_BLOB;
    idx[i] = j;
    dst[i] = total;
    total += align256(t.bytes);
  }

  mbt_model* m = new (std::nothrow) mbt_model();
  if (!m) return MBT_ERR_OOM;
  m->h = h;
  m->h.n_tensors = 0;
  m->h.table_offset = 0;
  m->device = dev;
  m->num_sms = prop.multiProcessorCount;
  m->wtype = fp8 ? W_E4M3 : W_BF16;
  m->kv8 = h.kv_dtype == MBT_DTYPE_E4M3;
  m->stream = stream_config(attn_smem_bytes((int)h.head_dim, m->kv8, (int)(h.n_q_heads / h.n_kv_heads)),
                            (int)(h.n_q_heads * h.head_dim));
  int rc = MBT_OK;
  if (gemv_init() != cudaSuccess || attn_init() != cudaSuccess) rc = MBT_ERR_CUDA;
  if (rc == MBT_OK && cudaMalloc(&m->wmem, total) != cudaSuccess) { cudaGetLastError(); rc = MBT_ERR_OOM; }
  if (rc == MBT_OK && cudaMalloc(&m->err, 256) != cudaSuccess) { cudaGetLastError(); rc = MBT_ERR_OOM; }
  const size_t rope_bytes = (size_t)h.max_pos * (h.head_dim / 2) * sizeof(float2);
  if (rc == MBT_OK && cudaMalloc(&m->rope, rope_bytes) != cudaSuccess) { cudaGetLastError(); rc = MBT_ERR_OOM; }
  if (rc != MBT_OK) { model_destroy(m); return rc; }
  m->wbytes = total;
  char* base = (char*)m->wmem;
  for (size_t i = 0; i < want.size() && rc == MBT_OK; ++i) {
    const mbt_blob_tensor& t = tab[idx[i]];
    const cudaMemcpyKind k = blob_is_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    if (cudaMemcpyAsync(base + dst[i], (const char*)blob + t.offset, t.bytes, k, s) != cudaSuccess) rc = MBT_ERR_CUDA;
  }
  if (rc == MBT_OK && cudaMemsetAsync(m->err, 0, 256, s) != cudaSuccess) rc = MBT_ERR_CUDA;
  // RoPE table: angle p * theta^(-2i/d), evaluated in double precision
  {
    const int half = (int)h.head_dim / 2;
    std::vector<float2> tabl((size_t)h.max_pos * half);
    for (uint32_t p = 0; p < h.max_pos; ++p)
      for (int i = 0; i < half; ++i) {
        const double ang = (double)p * std::pow((double)h.rope_theta, -2.0 * i / (double)h.head_dim);
        tabl[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    if (rc == MBT_OK && cudaMemcpyAsync(m->rope, tabl.data(), rope_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
      rc = MBT_ERR_CUDA;
    if (rc == MBT_OK && cudaStreamSynchronize(s) != cudaSuccess) rc = MBT_ERR_CUDA;
  }
  if (rc != MBT_OK) { model_destroy(m); return rc; }

  auto at = [&](uint32_t kind, int layer) -> void* {
    for (size_t i = 0; i < want.size(); ++i)
      if (want[i].kind == kind && want[i].layer == layer) return base + dst[i];
    return nullptr;
  };
  m->embed = (const bf16*)at(MBT_T_EMBED, -1);
  m->g_final = (const bf16*)at(MBT_T_G_FINAL, -1);
  m->lm = at(MBT_T_LM_HEAD, -1);
  m->s_lm = (const float*)at(MBT_T_S_LM, -1);
  m->layers.resize(h.n_layers);
  for (int l = 0; l < (int)h.n_layers; ++l) {
    Layer& L = m->layers[l];
    L.w_qkv = at(MBT_T_W_QKV, l); L.s_qkv = (const float*)at(MBT_T_S_QKV, l);
    L.w_o = at(MBT_T_W_O, l); L.s_o = (const float*)at(MBT_T_S_O, l);
    L.w_gu = at(MBT_T_W_GU, l); L.s_gu = (const float*)at(MBT_T_S_GU, l);
    L.w_down = at(MBT_T_W_DOWN, l); L.s_down = (const float*)at(MBT_T_S_DOWN, l);
    L.g_attn = (const bf16*)at(MBT_T_G_ATTN, l); L.g_ffn = (const bf16*)at(MBT_T_G_FFN, l);
  }
  // tensor maps for the tensor-core path (64-row boxes: BF16 tiles swizzled
  // for the MMA, e4m3 tiles plain for the widening warps)
  if (tc_init() == cudaSuccess) {
    const int Hh = (int)h.hidden, Qd = (int)(h.n_q_heads * h.head_dim), Ff = (int)h.ffn;
    const int QKVr = (int)((h.n_q_heads + 2 * h.n_kv_heads) * h.head_dim);
    auto mk = [&](TmaMap* map, const void* base, int rows, int K) {
      return (m->wtype == W_E4M3 ? tc_make_map_u8(map, base, rows, K, 64) : tc_make_map(map, base, rows, K, 64)) ==
             cudaSuccess;
    };
    m->wmaps.resize((size_t)h.n_layers * 4 + 1);
    bool ok = true;
    for (int l = 0; l < (int)h.n_layers && ok; ++l) {
      const Layer& L = m->layers[l];
      ok = mk(&m->wmaps[l * 4 + 0], L.w_qkv, QKVr, Hh) && mk(&m->wmaps[l * 4 + 1], L.w_o, Hh, Qd) &&
           mk(&m->wmaps[l * 4 + 2], L.w_gu, 2 * Ff, Hh) && mk(&m->wmaps[l * 4 + 3], L.w_down, Hh, Ff);
    }
    ok = ok && mk(&m->wmaps[(size_t)h.n_layers * 4], m->lm, (int)h.vocab, Hh);
    m->tc_ok = ok;
  }
  cudaGetLastError();
  *out = m;
  return MBT_OK;
}

int model_destroy(mbt_model* m) {
  if (!m) return MBT_OK;
  cudaDeviceSynchronize();
  destroy_graphs(m);
  free_ws(m->ws);
  free_ws(m->ws_eager);
  if (m->samp_z) cudaFree(m->samp_z);
  if (m->wmem) cudaFree(m->wmem);
  if (m->err) cudaFree(m->err);
  if (m->rope) cudaFree(m->rope);
  delete m;
  return MBT_OK;
}

int model_info(const mbt_model* m, mbt_blob_header* out) {
  if (!m || !out) return MBT_ERR_BAD_ARG;
  *out = m->h;
  return MBT_OK;
}

size_t kv_bytes(const mbt_model* m, int num_blocks) {
  if (!m || num_blocks < 1) return 0;
  return 2 * kv_layer_half_bytes(m, num_blocks) * m->h.n_layers;
}

int kv_alloc(mbt_model* m, int num_blocks, void* mem, mbt_kv** out) {
  if (!m || !out || num_blocks < 1) return MBT_ERR_BAD_ARG;
  *out = nullptr;
  mbt_kv* kv = new (std::nothrow) mbt_kv();
  if (!kv) return MBT_ERR_OOM;
  kv->m = m;
  kv->num_blocks = num_blocks;
  kv->bytes = kv_bytes(m, num_blocks);
  if (mem) {
    if ((uintptr_t)mem % 16) { delete kv; return MBT_ERR_BAD_ARG; }
    kv->pool = mem;
  } else {
    if (cudaMalloc(&kv->pool, kv->bytes) != cudaSuccess) { cudaGetLastError(); delete kv; return MBT_ERR_OOM; }
    kv->owned = true;
  }
  kv->k_scale.assign(m->h.n_layers, 1.0f);
  kv->v_scale.assign(m->h.n_layers, 1.0f);
  *out = kv;
  return MBT_OK;
}

int kv_free(mbt_kv* kv) {
  if (!kv) return MBT_OK;
  if (kv->m && kv->m->graph_kv == kv) destroy_graphs(kv->m);
  if (kv->owned && kv->pool) { cudaDeviceSynchronize(); cudaFree(kv->pool); }
  delete kv;
  return MBT_OK;
}

int kv_pool(const mbt_kv* kv, void** pool, size_t* bytes) {
  if (!kv || !pool || !bytes) return MBT_ERR_BAD_ARG;
  *pool = kv->pool;
  *bytes = kv->bytes;
  return MBT_OK;
}

int kv_set_scales(mbt_kv* kv, const float* ks, const float* vs) {
  if (!kv || !ks || !vs) return MBT_ERR_BAD_ARG;
  const int L = (int)kv->m->h.n_layers;
  for (int l = 0; l < L; ++l)
    if (!(ks[l] > 0.f) || !(vs[l] > 0.f) || !std::isfinite(ks[l]) || !std::isfinite(vs[l])) return MBT_ERR_BAD_ARG;
  kv->k_scale.assign(ks, ks + L);
  kv->v_scale.assign(vs, vs + L);
  if (kv->m->graph_kv == kv) destroy_graphs(kv->m);
  return MBT_OK;
}

int model_set_eager(mbt_model* m, int eager) {
  if (!m) return MBT_ERR_BAD_ARG;
  m->eager = eager ? 1 : 0;
  return MBT_OK;
}

int model_capture(mbt_model* m, mbt_kv* kv, const int* ladder, int n, int mbs, void* stream) {
  if (!m || !kv || kv->m != m || mbs < 1) return MBT_ERR_BAD_ARG;
  std::vector<int> rungs;
  if (ladder) {
    if (n < 1) return MBT_ERR_BAD_ARG;
    for (int i = 0; i < n; ++i) {
      if (ladder[i] < 1 || (i && ladder[i] <= ladder[i - 1])) return MBT_ERR_BAD_ARG;
      rungs.push_back(ladder[i]);
    }
  } else {
    rungs = {1, 2, 4};
    for (int r = 8; r <= 64; r += 8) rungs.push_back(r);
  }
  cudaStream_t s = (cudaStream_t)stream;
  destroy_graphs(m);
  const int Rmax = rungs.back();
  int rc = ensure_ws(m, m->ws, Rmax, mbs);
  if (rc != MBT_OK) return rc;
  // static input buffers
  size_t off = 0;
  auto take = [&](size_t b) { size_t o = off; off += align256(b); return o; };
  const size_t o_tok = take(Rmax * 4), o_pos = take(Rmax * 4), o_sl = take(Rmax * 4);
  const size_t o_bt = take((size_t)Rmax * mbs * 4), o_next = take(Rmax * 4);
  const size_t o_lg = take((size_t)Rmax * m->h.vocab * 4);
  if (cudaMalloc(&m->statics, off) != cudaSuccess) { cudaGetLastError(); return MBT_ERR_OOM; }
  char* b = (char*)m->statics;
  m->s_tok = (int*)(b + o_tok); m->s_pos = (int*)(b + o_pos); m->s_sl = (int*)(b + o_sl);
  m->s_bt = (int*)(b + o_bt); m->s_next = (int*)(b + o_next); m->s_logits = (float*)(b + o_lg);
  m->graph_mbs = mbs;

  cudaStream_t cs;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return MBT_ERR_CUDA;
  for (int R : rungs) {
    // all rows padding: token 0, position 0, the null block
    StageArgs st{0, R, nullptr, nullptr, nullptr, 1, nullptr, m->s_tok, m->s_pos, m->s_bt, mbs,
                 m->s_sl, kv->num_blocks, nullptr};
    if (launch_stage_inputs(st, s) != cudaSuccess) { rc = MBT_ERR_CUDA; break; }
    Plan p = make_plan(m, R, mbs);
    // warm-up run outside capture
    rc = run_step(m, m->ws, kv, p, m->s_tok, m->s_pos, m->s_bt, mbs, m->s_sl, m->s_next, m->s_logits, s);
    if (rc != MBT_OK) break;
    if (cudaStreamSynchronize(s) != cudaSuccess) { rc = MBT_ERR_CUDA; break; }
    Graph g;
    g.R = R;
    for (int v = 0; v < 2 && rc == MBT_OK; ++v) {
      cudaGraph_t graph;
      if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) { rc = MBT_ERR_CUDA; break; }
      int rr = run_step(m, m->ws, kv, p, m->s_tok, m->s_pos, m->s_bt, mbs, m->s_sl, m->s_next,
                        v ? m->s_logits : nullptr, cs);
      cudaError_t ce = cudaStreamEndCapture(cs, &graph);
      if (rr != MBT_OK || ce != cudaSuccess) { rc = MBT_ERR_CUDA; if (ce == cudaSuccess) cudaGraphDestroy(graph); break; }
      size_t nn = 0;
      cudaGraphGetNodes(graph, nullptr, &nn);
      g.nodes = (int)nn;
      if (cudaGraphInstantiate(&g.exec[v], graph, 0) != cudaSuccess) rc = MBT_ERR_CUDA;
      cudaGraphDestroy(graph);
    }
    if (rc != MBT_OK) {
      for (auto& e : g.exec) if (e) cudaGraphExecDestroy(e);
      break;
    }
    m->graphs.push_back(g);
  }
  cudaStreamDestroy(cs);
  if (rc != MBT_OK) { cudaGetLastError(); destroy_graphs(m); return rc; }
  if (cudaMemsetAsync(m->err, 0, 4, s) != cudaSuccess) return MBT_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MBT_ERR_CUDA;
  m->graph_kv = kv;
  return MBT_OK;
}

// The graph that serves B rows with block tables of bt_stride entries: the
// smallest captured rung >= B, provided the graphs are bound to this cache and
// their static table (graph_mbs entries per row) can hold the caller's table.
static const Graph* pick_graph(const mbt_model* m, const mbt_kv* kv, int B, int bt_stride) {
  if (m->eager || m->graph_kv != kv || bt_stride > m->graph_mbs) return nullptr;
  for (const Graph& g : m->graphs)
    if (g.R >= B) return &g;
  return nullptr;
}

int decode_step(mbt_model* m, mbt_kv* kv, int B, const int32_t* tok, const int32_t* pos,
                const int32_t* bt, int bt_stride, const int32_t* sl, int32_t* next_ids,
                float* logits, void* stream) {
  if (!m || !kv) return MBT_ERR_BAD_ARG;
  if (B <= 0) return MBT_ERR_BATCH;
  if (kv->m != m || !tok || !pos || !bt || !sl || !next_ids || bt_stride < 1) return MBT_ERR_BAD_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const Graph* g = pick_graph(m, kv, B, bt_stride);
  if (g) {
    // the staging kernel keeps the caller's table width: entries past
    // bt_stride are invalid ids, and a row whose seq_len needs more than
    // bt_stride blocks is flagged and attends over nothing, as it does eagerly
    StageArgs st{B, g->R, tok, pos, bt, bt_stride, sl, m->s_tok, m->s_pos, m->s_bt, m->graph_mbs,
                 m->s_sl, kv->num_blocks, m->err};
    MBT_CUDA(launch_stage_inputs(st, s));
    MBT_CUDA(cudaGraphLaunch(g->exec[logits ? 1 : 0], s));
    MBT_CUDA(cudaMemcpyAsync(next_ids, m->s_next, (size_t)B * 4, cudaMemcpyDeviceToDevice, s));
    if (logits)
      MBT_CUDA(cudaMemcpyAsync(logits, m->s_logits, (size_t)B * m->h.vocab * 4, cudaMemcpyDeviceToDevice, s));
    return MBT_OK;
  }
  // eager: the graph-bound workspace when it is large enough or no graph is
  // bound to it; otherwise a separate one, so that the graphs stay valid
  Workspace* w = &m->ws;
  if (!m->graphs.empty() && !ws_covers(m->ws, ws_need(m, m->ws, B, bt_stride))) w = &m->ws_eager;
  int rc = ensure_ws(m, *w, B, bt_stride);
  if (rc != MBT_OK) return rc;
  Plan p = make_plan(m, B, bt_stride);
  return run_step(m, *w, kv, p, tok, pos, bt, bt_stride, sl, next_ids, logits, s);
}

int decode_step_sample(mbt_model* m, mbt_kv* kv, int B, const int32_t* tok, const int32_t* pos,
                       const int32_t* bt, int bt_stride, const int32_t* sl, const mbt_sampling* sp,
                       int32_t* next_ids, float* logits, void* stream) {
  if (!m || !kv || !sp) return MBT_ERR_BAD_ARG;
  if (B <= 0) return MBT_ERR_BATCH;
  if (kv->m != m || !tok || !pos || !bt || !sl || !next_ids || bt_stride < 1) return MBT_ERR_BAD_ARG;
  if (!(sp->temperature > 0.f) || !std::isfinite(sp->temperature) || sp->top_k < 0 || sp->top_k > MBT_TOPK_MAX ||
      !(sp->top_p > 0.f) || !(sp->top_p <= 1.f))
    return MBT_ERR_BAD_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  SampleCfg smp = {};
  smp.gum.on = 1;
  smp.gum.inv_t = 1.0f / sp->temperature;
  smp.gum.seed_lo = (uint32_t)(sp->seed & 0xffffffffu); smp.gum.seed_hi = (uint32_t)(sp->seed >> 32);
  smp.gum.step_lo = (uint32_t)(sp->step & 0xffffffffu); smp.gum.step_hi = (uint32_t)(sp->step >> 32);
  const bool cut = sp->top_k > 0 || sp->top_p < 1.f;
  smp.mode = cut ? 2 : 1;
  smp.k = sp->top_k > 0 ? sp->top_k : kTopKMax;
  smp.top_p = sp->top_p;
  if (cut) {
    if (m->samp_rows < B) {
      if (cudaStreamSynchronize(s) != cudaSuccess) return MBT_ERR_CUDA;
      if (m->samp_z) cudaFree(m->samp_z);
      m->samp_z = nullptr;
      m->samp_rows = 0;
      if (cudaMalloc(&m->samp_z, (size_t)B * m->h.vocab * 4) != cudaSuccess) { cudaGetLastError(); return MBT_ERR_OOM; }
      m->samp_rows = B;
    }
    smp.z = m->samp_z;
  }
  Workspace* w = &m->ws;
  if (!m->graphs.empty() && !ws_covers(m->ws, ws_need(m, m->ws, B, bt_stride))) w = &m->ws_eager;
  int rc = ensure_ws(m, *w, B, bt_stride);
  if (rc != MBT_OK) return rc;
  Plan p = make_plan(m, B, bt_stride);
  return run_step(m, *w, kv, p, tok, pos, bt, bt_stride, sl, next_ids, logits, s, false, &smp);
}

int prefill(mbt_model* m, mbt_kv* kv, int n, const int32_t* tokens, int start_pos, const int32_t* block_table,
            int bt_len, int32_t* next_id, float* logits, void* stream) {
  if (!m || !kv) return MBT_ERR_BAD_ARG;
  if (n < 1) return MBT_ERR_BATCH;
  if (kv->m != m || !tokens || !block_table || !next_id || bt_len < 1 || start_pos < 0) return MBT_ERR_BAD_ARG;
  const long long end = (long long)start_pos + n;
  if (end > (long long)m->h.max_pos || end > (long long)bt_len * kBlockTokens) return MBT_ERR_BAD_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int C = std::min(n, kPrefillChunk);
  Workspace* w = &m->ws;
  if (!m->graphs.empty() && !ws_covers(m->ws, ws_need(m, m->ws, C, bt_len))) w = &m->ws_eager;
  int rc = ensure_ws(m, *w, C, bt_len);
  if (rc != MBT_OK) return rc;
  for (int c0 = 0; c0 < n; c0 += C) {
    const int R = std::min(C, n - c0);
    const bool last = c0 + R == n;
    PrefillStageArgs st{R, tokens + c0, start_pos + c0, block_table, bt_len, w->pf_tok, w->pf_pos, w->pf_sl, w->pf_bt};
    MBT_CUDA(launch_stage_prefill(st, s));
    const Plan p = make_plan(m, R, bt_len);
    rc = run_step(m, *w, kv, p, w->pf_tok, w->pf_pos, w->pf_bt, bt_len, w->pf_sl, last ? next_id : nullptr,
                  last ? logits : nullptr, s, true);
    if (rc != MBT_OK) return rc;
  }
  return MBT_OK;
}

int model_poll_errors(mbt_model* m, void* stream, uint32_t* bits) {
  if (!m || !bits) return MBT_ERR_BAD_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t v = 0;
  MBT_CUDA(cudaStreamSynchronize(s));
  MBT_CUDA(cudaMemcpy(&v, m->err, 4, cudaMemcpyDeviceToHost));
  MBT_CUDA(cudaMemset(m->err, 0, 4));
  *bits = v;
  return MBT_OK;
}

int model_stats(mbt_model* m, int B, int* kernels, int* uses_graph) {
  if (!m || !kernels || !uses_graph || B < 1) return MBT_ERR_BAD_ARG;
  const Graph* g = pick_graph(m, m->graph_kv, B, m->graph_mbs);
  if (g) {
    *kernels = g->nodes + 1;   // graph kernel nodes + the staging kernel
    *uses_graph = 1;
  } else {
    *kernels = make_plan(m, B, std::max(1, m->graph_mbs)).kernels;
    *uses_graph = 0;
  }
  return MBT_OK;
}

}  // extern "C"
