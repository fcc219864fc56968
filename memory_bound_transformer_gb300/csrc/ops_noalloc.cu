// Paged attention that allocates nothing: the split-K partials, the (max, sum)
// pairs and the merge tickets live in one file-scope device array of
// MBT_NOALLOC_SCRATCH_BYTES.
//
// Some callers cannot allocate device memory at the moment they run attention:
// serving processes that reserve almost all HBM for their KV pool up front (a
// new allocation would fail or fragment that reservation), latency-critical
// paths where cudaMalloc / cudaFree may synchronise the device, and runtimes
// whose allocator policy forbids allocation after start-up. This entry point
// serves them.
//
// Every call shares the array, and it keeps the previous call's contents, so
// calls that overlap on the GPU (on different streams, or from several host
// threads) race with one another; issue them in one stream order. The first
// call on a device fetches the array's device address (set-up, once per
// device); make that first call before any stream capture.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "../../include/mbt_ops.h"

using namespace mbt;

namespace {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kScratchBytes = MBT_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};   // device address of g_attn_scratch, per device
bool g_ready[kMaxDevices] = {};

// Set-up, once per device with that device current: the host-side name of the
// array is only a stand-in, so fetch its device address.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MBT_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ready[dev]) {
    if (gemv_init() != cudaSuccess || attn_init() != cudaSuccess) return MBT_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return MBT_ERR_CUDA;
    g_ptr[dev] = p;
    g_ready[dev] = true;
  }
  *out = g_ptr[dev];
  return MBT_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" {

size_t op_paged_attention_noalloc_limit(void) { return kScratchBytes; }

int op_paged_attention_noalloc(int B, const float* q, int nq, int nkv, int d, const void* kpool,
                               const void* vpool, int kv_dtype, float k_scale, float v_scale,
                               const int32_t* bt, int bt_stride, const int32_t* seq_lens,
                               int num_blocks, float* out, uint32_t* err, void* stream) {
  if (B < 1 || !q || nq < 1 || nkv < 1 || nq % nkv || nq / nkv > 16 || (d != 64 && d != 128) ||
      !kpool || !vpool || !bt || bt_stride < 1 || !seq_lens || num_blocks < 1 || !out ||
      (kv_dtype != MBT_DTYPE_BF16 && kv_dtype != MBT_DTYPE_E4M3))
    return MBT_ERR_BAD_ARG;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MBT_ERR_NO_DEVICE;
  AttnArgs a = {};
  a.B = B; a.q = q; a.nq = nq; a.nkv = nkv; a.d = d; a.kpool = kpool; a.vpool = vpool;
  a.kv_fp8 = kv_dtype == MBT_DTYPE_E4M3; a.k_scale = k_scale; a.v_scale = v_scale;
  a.bt = bt; a.bt_stride = bt_stride; a.seq_lens = seq_lens; a.num_blocks = num_blocks;
  attn_plan(B, nkv, bt_stride, nsm, attn_ctas_per_sm(a.kv_fp8, nq / nkv), &a.bps, &a.nsplit);
  a.out = out; a.err = err;
  const size_t heads = (size_t)B * nq * a.nsplit;
  const size_t b_po = align256(heads * d * sizeof(float));
  const size_t b_ml = align256(heads * sizeof(float2));
  const size_t b_tk = (size_t)B * nkv * sizeof(int);
  if (b_po + b_ml + b_tk > kScratchBytes) return MBT_ERR_SCRATCH;
  void* base = nullptr;
  int rc = scratch_for_current_device(&base);
  if (rc != MBT_OK) return rc;
  char* p = (char*)base;
  a.part_o = (float*)p;
  a.part_ml = (float2*)(p + b_po);
  a.tickets = (int*)(p + b_po + b_ml);
  cudaStream_t s = (cudaStream_t)stream;
  // the array keeps the previous call's contents: the tickets must start at zero
  if (cudaMemsetAsync(a.tickets, 0, b_tk, s) != cudaSuccess) return MBT_ERR_CUDA;
  return launch_attention(a, s) == cudaSuccess ? MBT_OK : MBT_ERR_CUDA;
}

}  // extern "C"
