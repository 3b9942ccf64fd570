// attn_bwd_noalloc: the attention backward for callers that cannot give the
// library a workspace buffer.
//
// Who needs this: code that is handed only its input and output buffers and is
// not allowed to allocate device memory itself, such as a plug-in whose host
// framework owns every device allocation, or a latency-critical loop that must
// not call cudaMalloc after start-up (cudaMalloc can synchronise the device).
// attn_bwd needs a caller-provided workspace (the row statistic D and an fp32
// dq accumulator); this entry point instead uses a fixed scratch array that
// lives in the library's own device memory.
//
// The scratch array is a file-scope __device__ array of ATTN_NOALLOC_SCRATCH_BYTES
// (32 MiB). Every GPU that loads the library holds it until the process exits.
// In host code its name is only a host-side stand-in, never a device address,
// so the first call on each device looks up the real address with
// cudaGetSymbolAddress (with that device current) and caches it together with
// the id of the device's context; a later call in a different context (after
// cudaDeviceReset, say, when the module is loaded anew and the array may move)
// looks it up again. Make the first call on a device before any stream
// capture. Nothing here calls cudaMalloc, cudaFree or an allocating library
// routine.
//
// All calls share the one array and it keeps the previous call's contents: the
// backward's pre-pass zeroes the dq accumulator and rewrites D on every call,
// so stale contents never leak into a result. Calls whose GPU work overlaps
// (different streams, or several host threads) race on the array; issue them
// in order on one stream.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace attn {
bool current_context_id(unsigned long long* id);   // attn_api.cu
}

namespace {

constexpr size_t kScratchBytes = ATTN_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
struct Cached {
  unsigned long long ctx = 0;   // id of the context the address belongs to
  void* addr = nullptr;
};
Cached g_scratch[kMaxDevices];

// Device address of the scratch array in the current device's context (looked
// up once per context).
attn_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  Cached& c = g_scratch[dev];
  unsigned long long id = 0;
  if (!c.addr || !attn::current_context_id(&id) || id != c.ctx) {
    void* p = nullptr;   // the lookup makes the device's primary context current if none is
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    if (!attn::current_context_id(&id)) return ATTN_ERR_CUDA;
    c.addr = p;
    c.ctx = id;
  }
  *out = c.addr;
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_bwd_noalloc(const void* dout, const void* qkv, const void* out,
                                          const float* lse, void* dqkv, int B, int T, int C, int NH,
                                          int causal, attn_dtype_t dtype, void* stream) {
  const size_t need = attn_bwd_workspace_size(B, T, C, NH, causal, dtype);
  if (need > kScratchBytes) return ATTN_ERR_WORKSPACE;   // problem too large for the fixed scratch
  void* scratch = nullptr;
  if (need > 0) {
    const attn_status_t st = scratch_address(&scratch);
    if (st != ATTN_OK) return st;
  }
  // need == 0 means attn_bwd rejects the arguments; it reports why.
  return attn_bwd(dout, qkv, out, lse, dqkv, B, T, C, NH, causal, dtype, scratch, kScratchBytes, stream);
}
