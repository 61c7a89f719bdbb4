// tv_verify_greedy_static: greedy verification without a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the point where they call
// the library - for example a plugin whose host framework plans and owns every device
// buffer up front, code that runs while another component is capturing a CUDA graph
// and forbids allocations, or runtimes that disallow allocation after start-up.  They
// still pass their own inputs and outputs; only the vocab pass's scratch (per-split row
// partials, per-row results and the completion counters) moves into a fixed array that
// lives in this library's device image.
//
// The array is a file-scope __device__ object of kStaticScratchBytes: every GPU that
// loads the library holds it until the process exits.  Host code may not use its name as
// a device address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and clears the array once; later calls
// reuse the cached address.  All calls share the one array, so calls that overlap on the
// GPU (different streams, or concurrent host threads) race on it.
#include <mutex>

#include "tv_kernels.cuh"

namespace tv {

constexpr size_t kStaticScratchBytes = 4u << 20;  // 4 MiB per device

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};

// Address of g_static_scratch on the current device; the first call per device also
// zero-fills it (a synchronous memset, no allocation).
cudaError_t static_scratch_ptr(void** out) {
  int devid = 0;
  cudaError_t e = cudaGetDevice(&devid);
  if (e != cudaSuccess) return e;
  if (devid < 0 || devid >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[devid]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    e = cudaMemset(p, 0, kStaticScratchBytes);
    if (e != cudaSuccess) return e;
    g_ptr[devid] = p;
  }
  *out = g_ptr[devid];
  return cudaSuccess;
}

}  // namespace
}  // namespace tv

using namespace tv;

extern "C" TV_API tv_status tv_verify_greedy_static(const void* logits, const int32_t* parent, const int32_t* tokens,
                                                    int B, int N, int V, tv_dtype dtype, int32_t* accepted_nodes,
                                                    int32_t* accept_len, int32_t* bonus_token, float* p_draft,
                                                    float* row_lse, int32_t* row_argmax, int32_t* dev_status,
                                                    tv_stream_t stream) {
  if (!logits || !parent || !tokens || !accepted_nodes || !accept_len || !bonus_token) return TV_ERR_NULL;
  if (dtype != TV_F32 && dtype != TV_BF16) return TV_ERR_DTYPE;
  if (B < 1 || N < 1 || N > kMaxNodes || V < 1) return TV_ERR_SHAPE;
  const long long rows = (long long)B * N;
  if (rows > 0x7fffffffLL || (long long)N * V > 0x7fffffffLL) return TV_ERR_SHAPE;
  if (rows > kMaxVerifyRows) return TV_ERR_SHAPE;
  VerifyWs w;
  const size_t need = verify_ws_layout(B, N, V, 0, &w);
  if (need > kStaticScratchBytes) return TV_ERR_WORKSPACE;  // the fixed array is too small
  void* scratch = nullptr;
  if (static_scratch_ptr(&scratch) != cudaSuccess) return TV_ERR_CUDA;
  char* ws = reinterpret_cast<char*>(scratch);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the completion counters must start at zero; clear them on the caller's stream
  if (cudaMemsetAsync(ws + w.row_cnt, 0, w.part - w.row_cnt, s) != cudaSuccess) return TV_ERR_CUDA;
  return launch_vocab_pass(logits, nullptr, parent, tokens, B, N, V, dtype, 1.0f, ws, w, accepted_nodes, accept_len,
                           bonus_token, p_draft, nullptr, row_lse, row_argmax, nullptr, dev_status, 0,
                           s) == cudaSuccess
             ? TV_OK
             : TV_ERR_CUDA;
}
