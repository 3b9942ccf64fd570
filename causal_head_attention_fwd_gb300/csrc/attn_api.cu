// C ABI of the attention library: argument checks, TMA descriptor encoding,
// kernel dispatch and the device error word. Declared in include/attn.h.
#include <cstdint>
#include <cstring>
#include <cmath>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/attn.h"
#include "common.cuh"

namespace attn {

// Declared in the kernel translation units.
cudaError_t launch_fwd_bf16(const CUtensorMap& map_qkv, const CUtensorMap& map_out, float* lse,
                            const Problem& pr, cudaStream_t stream);
cudaError_t launch_bwd_bf16(const CUtensorMap& map_qkv, const CUtensorMap& map_dout,
                            const CUtensorMap& map_dqkv, const CUtensorMap& map_dqacc, const void* dout,
                            const void* out, const float* lse, void* dqkv, float* ws_D, float* ws_dq,
                            const Problem& pr, cudaStream_t stream);
int fwd_schedule(const Problem& pr, int n_cta, int* off, int* items, int cap);
cudaError_t launch_fwd_f32(const CUtensorMap& map_q_l, const CUtensorMap& map_q_s, const CUtensorMap& map_out_l,
                           float* lse, const Problem& pr, cudaStream_t stream);
cudaError_t launch_bwd_f32(const CUtensorMap& map_q_l, const CUtensorMap& map_q_s, const CUtensorMap& map_do_l,
                           const CUtensorMap& map_do_s, const CUtensorMap& map_g_l, const float* dout,
                           const float* out, const float* lse, float* ws_D, const Problem& pr,
                           cudaStream_t stream);

cudaError_t launch_fwd_fp8(const CUtensorMap& map_qkv, const CUtensorMap& map_out, const float* descale, float* lse,
                           const Problem& pr, cudaStream_t stream);
cudaError_t launch_fp8_dequant(const void* codes, const float* descale, void* out, int B, int T, int C, int NH,
                               cudaStream_t stream);
cudaError_t launch_linear(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                          const void* bias, int M, int N, int K, cudaStream_t stream);
cudaError_t launch_att(const CUtensorMap& map_qkv, const CUtensorMap& map_pre, const CUtensorMap& map_att, bool tma_out,
                       const float* lse, float* preatt, float* att, bool f32, const Problem& pr, cudaStream_t stream);

size_t decode_workspace_bytes(int B, int L, int C, int NH, int Tq, bool f32);
int decode_max_tq();
int decode_chunk(bool f32);
cudaError_t launch_decode(const CUtensorMap& map_qkv, const CUtensorMap& map_kq, const CUtensorMap& map_q,
                          const void* qkv, void* out, float* lse, float* part, bool f32, int B, int L, int C, int NH,
                          int Tq, cudaStream_t stream);

static __device__ int g_error_word = 0;

static constexpr int kMaxDevices = 64;
static std::mutex g_mu;

// Id of the calling thread's current CUDA context, unique for the life of the
// process (a context made after cudaDeviceReset gets a new one, even if its
// handle value is reused). False when no context is current or the driver
// entry point is unavailable.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetId_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  return fn && fn(nullptr, id) == CUDA_SUCCESS;
}

// The device address of a __device__ symbol is a property of the module loaded
// into one context: it is looked up once per device and looked up again when
// that device's context has changed (after cudaDeviceReset the module is
// loaded anew and the symbol may move).
struct SymbolAddr {
  unsigned long long ctx = 0;
  int* addr = nullptr;
};
static SymbolAddr g_error_addr[kMaxDevices];

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  unsigned long long id = 0;
  SymbolAddr& c = g_error_addr[dev];
  if (!c.addr || !current_context_id(&id) || id != c.ctx) {
    void* p = nullptr;   // the lookup makes the device's primary context current if none is
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess || !current_context_id(&id)) return nullptr;
    c.addr = static_cast<int*>(p);
    c.ctx = id;
  }
  return c.addr;
}

static int g_sm_count[kMaxDevices] = {0};

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

// ---------------------------------------------------------------- profiling
struct ProfState {
  bool enabled = false;
  struct Pending { cudaEvent_t a, b; };
  std::vector<Pending> pending[K_COUNT];
  std::vector<cudaEvent_t> pool;
  double total_ms[K_COUNT] = {};
  long long count[K_COUNT] = {};
  cudaEvent_t cur_begin[K_COUNT] = {};
};
static ProfState g_prof;

static cudaEvent_t take_event() {
  if (!g_prof.pool.empty()) {
    cudaEvent_t e = g_prof.pool.back();
    g_prof.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

void profile_begin(KernelId k, cudaStream_t s) {
  if (!g_prof.enabled) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t e = take_event();
  if (e && cudaEventRecord(e, s) == cudaSuccess) g_prof.cur_begin[k] = e;
}

void profile_end(KernelId k, cudaStream_t s) {
  if (!g_prof.enabled) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t a = g_prof.cur_begin[k];
  g_prof.cur_begin[k] = nullptr;
  if (!a) return;
  cudaEvent_t b = take_event();
  if (b && cudaEventRecord(b, s) == cudaSuccess) g_prof.pending[k].push_back({a, b});
}

// Resolve every pending event pair of kernel k into the running totals.
static bool profile_drain(int k) {
  for (auto& pe : g_prof.pending[k]) {
    if (cudaEventSynchronize(pe.b) != cudaSuccess) return false;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, pe.a, pe.b) != cudaSuccess) return false;
    g_prof.total_ms[k] += ms;
    g_prof.count[k] += 1;
    g_prof.pool.push_back(pe.a);
    g_prof.pool.push_back(pe.b);
  }
  g_prof.pending[k].clear();
  return true;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over a (B, T, W) row-major tensor of `esize`-byte elements, box
// {box_x, box_y, 1}. Rows past T read as zero; stores past T are dropped.
static bool encode_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int W, int T,
                      int B, int box_x, int box_y, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)W, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)W * esize, (cuuint64_t)W * esize * (cuuint64_t)T};
  cuuint32_t box[3] = {(cuuint32_t)box_x, (cuuint32_t)box_y, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static attn_status_t check_shape(int B, int T, int C, int NH, int causal, attn_dtype_t dtype) {
  if (B < 1 || T < 1 || C < 1 || NH < 1) return ATTN_ERR_INVALID_ARG;
  if (C % NH != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  const int hs = C / NH;
  if (hs != 32 && hs != 64) return ATTN_ERR_UNSUPPORTED;
  // element counts must fit the 32-bit grid/tile arithmetic of the kernels
  const double n3 = (double)B * T * 3.0 * C;
  if (n3 > 9.0e15 || (double)T > 2.0e9 || (double)B * NH * ((T + 255) / 256) > 2.0e9)
    return ATTN_ERR_INVALID_ARG;
  // the fp32 backward launches one CTA per (b, h, 128-row tile)
  if (dtype == ATTN_F32 && (double)B * NH * ((T + 127) / 128) > 2.0e9) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

static size_t esize(attn_dtype_t dt) { return dt == ATTN_BF16 ? 2 : 4; }

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace attn

using namespace attn;

extern "C" const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG: invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: head size or dtype not implemented";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED: pointer not 16-byte aligned";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE: workspace missing or too small";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: CUDA call or launch failed";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a kernel's bounded wait expired";
    case ATTN_ERR_BOUNDS: return "ATTN_ERR_BOUNDS: a kernel index check failed (debug build)";
  }
  return "ATTN_ERR_UNKNOWN";
}

extern "C" attn_status_t attn_fwd(const void* qkv, void* out, float* lse, int B, int T, int C, int NH,
                                  int causal, attn_dtype_t dtype, void* stream) {
  attn_status_t st = check_shape(B, T, C, NH, causal, dtype);
  if (st != ATTN_OK) return st;
  if (!qkv || !out || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(out) || !aligned16(lse)) return ATTN_ERR_MISALIGNED;
  const size_t e = esize(dtype);
  if (overlaps(out, (size_t)B * T * C * e, qkv, (size_t)B * T * 3 * C * e) ||
      overlaps(lse, (size_t)B * NH * T * 4, qkv, (size_t)B * T * 3 * C * e) ||
      overlaps(lse, (size_t)B * NH * T * 4, out, (size_t)B * T * C * e))
    return ATTN_ERR_INVALID_ARG;
  Problem pr{B, T, C, NH, C / NH, causal};
  if (!device_error_word() || device_sm_count() <= 0) return ATTN_ERR_CUDA;
  if (dtype == ATTN_F32) {
    // fp32 tiles: 32-column (128-byte) boxes, 128- or 64-row
    const CUtensorMapDataType f = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const CUtensorMapSwizzle w = CU_TENSOR_MAP_SWIZZLE_128B;
    CUtensorMap ql, qs, ol;
    if (!encode_3d(&ql, qkv, f, 4, 3 * C, T, B, 32, 128, w) || !encode_3d(&qs, qkv, f, 4, 3 * C, T, B, 32, 64, w) ||
        !encode_3d(&ol, out, f, 4, C, T, B, 32, 128, w))
      return ATTN_ERR_CUDA;
    cudaError_t ce = launch_fwd_f32(ql, qs, ol, lse, pr, static_cast<cudaStream_t>(stream));
    return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  const CUtensorMapSwizzle swz = pr.hs == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap mq, mo;
  if (!encode_3d(&mq, qkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 3 * C, T, B, pr.hs, BM, swz) ||
      !encode_3d(&mo, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, T, B, pr.hs, BM, swz))
    return ATTN_ERR_CUDA;
  cudaError_t ce = launch_fwd_bf16(mq, mo, lse, pr, static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" int attn_fwd_schedule(int B, int T, int C, int NH, int n_cta, int* off, int* items, int cap) {
  if (check_shape(B, T, C, NH, 1, ATTN_BF16) != ATTN_OK || n_cta < 1 || !off || !items || cap < 0) return -1;
  Problem pr{B, T, C, NH, C / NH, 1};
  return fwd_schedule(pr, n_cta, off, items, cap);
}

// Bytes of the FP8 descale array: 3 (q, k, v) x B*NH heads x ceil(T/128) row tiles, fp32.
static size_t fp8_descale_bytes(int B, int T, int NH) { return (size_t)3 * B * NH * ((T + BM - 1) / BM) * 4; }

extern "C" attn_status_t attn_fwd_fp8(const void* qkv, const float* descale, void* out, float* lse, int B, int T,
                                      int C, int NH, int causal, void* stream) {
  attn_status_t st = check_shape(B, T, C, NH, causal, ATTN_BF16);
  if (st != ATTN_OK) return st;
  if (!qkv || !descale || !out || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(out) || !aligned16(lse) || (reinterpret_cast<uintptr_t>(descale) & 3u))
    return ATTN_ERR_MISALIGNED;
  const size_t nq = (size_t)B * T * 3 * C, no = (size_t)B * T * C * 2, nl = (size_t)B * NH * T * 4;
  const size_t nd = fp8_descale_bytes(B, T, NH);
  if (overlaps(out, no, qkv, nq) || overlaps(lse, nl, qkv, nq) || overlaps(lse, nl, out, no) ||
      overlaps(descale, nd, out, no) || overlaps(descale, nd, lse, nl))
    return ATTN_ERR_INVALID_ARG;
  Problem pr{B, T, C, NH, C / NH, causal};
  if (!device_error_word() || device_sm_count() <= 0) return ATTN_ERR_CUDA;
  // e4m3 tiles: hs-byte rows (64- or 32-byte swizzle); bf16 output as in attn_fwd
  const CUtensorMapSwizzle s8 = pr.hs == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  const CUtensorMapSwizzle s16 = pr.hs == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap mq, mo;
  if (!encode_3d(&mq, qkv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 3 * C, T, B, pr.hs, BM, s8) ||
      !encode_3d(&mo, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, T, B, pr.hs, BM, s16))
    return ATTN_ERR_CUDA;
  cudaError_t ce = launch_fwd_fp8(mq, mo, descale, lse, pr, static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" attn_status_t attn_linear_fwd(const void* inp, const void* weight, const void* bias, void* out, int M,
                                         int N, int K, void* stream) {
  if (M < 1 || N < 1 || K < 1) return ATTN_ERR_INVALID_ARG;
  if (N % 8 != 0 || K % 8 != 0) return ATTN_ERR_UNSUPPORTED;     // 16-byte row strides for the tensor copies
  if ((double)((M + 127) / 128) * ((N + 255) / 256) > 2.0e9) return ATTN_ERR_INVALID_ARG;   // tile count fits an int
  if (!inp || !weight || !out) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(inp) || !aligned16(weight) || !aligned16(out) || (bias && !aligned16(bias)))
    return ATTN_ERR_MISALIGNED;
  const size_t ni = (size_t)M * K * 2, nw = (size_t)N * K * 2, no = (size_t)M * N * 2, nb = (size_t)N * 2;
  if (overlaps(out, no, inp, ni) || overlaps(out, no, weight, nw) || (bias && overlaps(out, no, bias, nb)))
    return ATTN_ERR_INVALID_ARG;
  if (!device_error_word() || device_sm_count() <= 0) return ATTN_ERR_CUDA;
  CUtensorMap ma, mb, mo;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle w = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!encode_3d(&ma, inp, bf, 2, K, M, 1, 64, 128, w) || !encode_3d(&mb, weight, bf, 2, K, N, 1, 64, 256, w) ||
      !encode_3d(&mo, out, bf, 2, N, M, 1, 64, 128, w))
    return ATTN_ERR_CUDA;
  cudaError_t ce = launch_linear(ma, mb, mo, bias, M, N, K, static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// FP8 backward scratch: the bf16 expansion of qkv (B*T*3C*2 bytes, 256-byte
// aligned), then attn_bwd's own bf16 workspace.
static size_t fp8_qkv_bytes(int B, int T, int C) { return (((size_t)B * T * 3 * C * 2) + 255) & ~(size_t)255; }

extern "C" size_t attn_bwd_fp8_workspace_size(int B, int T, int C, int NH, int causal) {
  if (check_shape(B, T, C, NH, causal, ATTN_BF16) != ATTN_OK) return 0;
  return fp8_qkv_bytes(B, T, C) + attn_bwd_workspace_size(B, T, C, NH, causal, ATTN_BF16);
}

extern "C" attn_status_t attn_bwd_fp8(const void* dout, const void* qkv, const float* descale, const void* out,
                                      const float* lse, void* dqkv, int B, int T, int C, int NH, int causal,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  attn_status_t st = check_shape(B, T, C, NH, causal, ATTN_BF16);
  if (st != ATTN_OK) return st;
  if (!dout || !qkv || !descale || !out || !lse || !dqkv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(qkv) || !aligned16(out) || !aligned16(lse) || !aligned16(dqkv) ||
      (reinterpret_cast<uintptr_t>(descale) & 3u))
    return ATTN_ERR_MISALIGNED;
  const size_t need = attn_bwd_fp8_workspace_size(B, T, C, NH, causal);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_MISALIGNED;
  const size_t n8 = (size_t)B * T * 3 * C, n3 = n8 * 2, n1 = (size_t)B * T * C * 2, nl = (size_t)B * NH * T * 4;
  const size_t nd = fp8_descale_bytes(B, T, NH);
  if (overlaps(dqkv, n3, qkv, n8) || overlaps(dqkv, n3, out, n1) || overlaps(dqkv, n3, dout, n1) ||
      overlaps(dqkv, n3, lse, nl) || overlaps(dqkv, n3, descale, nd) || overlaps(workspace, need, qkv, n8) ||
      overlaps(workspace, need, out, n1) || overlaps(workspace, need, dout, n1) ||
      overlaps(workspace, need, lse, nl) || overlaps(workspace, need, descale, nd) ||
      overlaps(workspace, need, dqkv, n3))
    return ATTN_ERR_INVALID_ARG;
  if (!device_error_word() || device_sm_count() <= 0) return ATTN_ERR_CUDA;
  // 1. the e4m3 codes expanded to bf16 values code * descale (the matmuls of the
  //    backward run in bf16), 2. the bf16 backward on them
  char* ws = static_cast<char*>(workspace);
  void* qkv16 = ws;
  if (launch_fp8_dequant(qkv, descale, qkv16, B, T, C, NH, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const size_t off = fp8_qkv_bytes(B, T, C);
  return attn_bwd(dout, qkv16, out, lse, dqkv, B, T, C, NH, causal, ATTN_BF16, ws + off, workspace_bytes - off,
                  stream);
}

extern "C" size_t attn_bwd_workspace_size(int B, int T, int C, int NH, int causal, attn_dtype_t dtype) {
  if (check_shape(B, T, C, NH, causal, dtype) != ATTN_OK) return 0;
  // D (B*NH*T fp32) rounded to 256 bytes; bf16 adds the fp32 dq accumulator
  // (B*T*C); the fp32 path writes dq straight into dqkv
  const size_t d_bytes = (((size_t)B * NH * T * 4) + 255) & ~(size_t)255;
  if (dtype == ATTN_F32) return d_bytes;
  return d_bytes + (size_t)B * T * C * 4;
}

extern "C" attn_status_t attn_bwd(const void* dout, const void* qkv, const void* out, const float* lse,
                                  void* dqkv, int B, int T, int C, int NH, int causal, attn_dtype_t dtype,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  attn_status_t st = check_shape(B, T, C, NH, causal, dtype);
  if (st != ATTN_OK) return st;
  if (!dout || !qkv || !out || !lse || !dqkv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(qkv) || !aligned16(out) || !aligned16(lse) || !aligned16(dqkv))
    return ATTN_ERR_MISALIGNED;
  const size_t need = attn_bwd_workspace_size(B, T, C, NH, causal, dtype);
  if (need > 0 && (!workspace || workspace_bytes < need)) return ATTN_ERR_WORKSPACE;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTN_ERR_MISALIGNED;
  const size_t e = esize(dtype);
  const size_t n3 = (size_t)B * T * 3 * C * e, n1 = (size_t)B * T * C * e, nl = (size_t)B * NH * T * 4;
  if (overlaps(dqkv, n3, qkv, n3) || overlaps(dqkv, n3, out, n1) || overlaps(dqkv, n3, dout, n1) ||
      overlaps(dqkv, n3, lse, nl))
    return ATTN_ERR_INVALID_ARG;
  // the workspace (D and the dq accumulator) is written: it may share no byte with any other buffer
  if (workspace && (overlaps(workspace, need, dqkv, n3) || overlaps(workspace, need, qkv, n3) ||
                    overlaps(workspace, need, out, n1) || overlaps(workspace, need, dout, n1) ||
                    overlaps(workspace, need, lse, nl)))
    return ATTN_ERR_INVALID_ARG;
  Problem pr{B, T, C, NH, C / NH, causal};
  if (!device_error_word() || device_sm_count() <= 0) return ATTN_ERR_CUDA;
  if (dtype == ATTN_F32) {
    const CUtensorMapDataType f = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const CUtensorMapSwizzle w = CU_TENSOR_MAP_SWIZZLE_128B;
    CUtensorMap ql, qs, dl, ds, gl;
    if (!encode_3d(&ql, qkv, f, 4, 3 * C, T, B, 32, 128, w) || !encode_3d(&qs, qkv, f, 4, 3 * C, T, B, 32, 64, w) ||
        !encode_3d(&dl, dout, f, 4, C, T, B, 32, 128, w) || !encode_3d(&ds, dout, f, 4, C, T, B, 32, 64, w) ||
        !encode_3d(&gl, dqkv, f, 4, 3 * C, T, B, 32, 128, w))
      return ATTN_ERR_CUDA;
    cudaError_t ce = launch_bwd_f32(ql, qs, dl, ds, gl, static_cast<const float*>(dout),
                                    static_cast<const float*>(out), lse, static_cast<float*>(workspace), pr,
                                    static_cast<cudaStream_t>(stream));
    return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  const CUtensorMapSwizzle swz = pr.hs == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap mq, md, mg;
  if (!encode_3d(&mq, qkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 3 * C, T, B, pr.hs, BM, swz) ||
      !encode_3d(&md, dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, T, B, pr.hs, BM, swz) ||
      !encode_3d(&mg, dqkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 3 * C, T, B, pr.hs, BM, swz))
    return ATTN_ERR_CUDA;
  float* ws_D = static_cast<float*>(workspace);
  float* ws_dq = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          ((((size_t)B * NH * T * 4) + 255) & ~(size_t)255));
  // fp32 dq accumulator (B, T, C): 32-column boxes (128 bytes) for the 128-byte swizzle
  CUtensorMap ma;
  if (!encode_3d(&ma, ws_dq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, T, B, 32, BM, CU_TENSOR_MAP_SWIZZLE_128B))
    return ATTN_ERR_CUDA;
  cudaError_t ce = launch_bwd_bf16(mq, md, mg, ma, dout, out, lse, dqkv, ws_D, ws_dq, pr,
                                   static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" attn_status_t attn_fwd_att(const void* qkv, const float* lse, float* preatt, float* att, int B, int T,
                                      int C, int NH, int causal, attn_dtype_t dtype, void* stream) {
  attn_status_t st = check_shape(B, T, C, NH, causal, dtype);
  if (st != ATTN_OK) return st;
  if (!qkv || !lse || (!preatt && !att)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(lse) || (preatt && !aligned16(preatt)) || (att && !aligned16(att)))
    return ATTN_ERR_MISALIGNED;
  const long long nt = (T + 127) / 128;
  if ((double)B * NH * (double)nt * (double)nt > 2.0e9) return ATTN_ERR_INVALID_ARG;
  const size_t e = esize(dtype);
  const size_t nq = (size_t)B * T * 3 * C * e, nl = (size_t)B * NH * T * 4, na = (size_t)B * NH * T * (size_t)T * 4;
  if ((preatt && (overlaps(preatt, na, qkv, nq) || overlaps(preatt, na, lse, nl))) ||
      (att && (overlaps(att, na, qkv, nq) || overlaps(att, na, lse, nl))) ||
      (preatt && att && overlaps(preatt, na, att, na)))
    return ATTN_ERR_INVALID_ARG;
  Problem pr{B, T, C, NH, C / NH, causal};
  if (!device_error_word()) return ATTN_ERR_CUDA;
  CUtensorMap mq;
  const bool f32 = dtype == ATTN_F32;
  const bool enc = f32 ? encode_3d(&mq, qkv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 3 * C, T, B, 32, BM,
                                   CU_TENSOR_MAP_SWIZZLE_128B)
                       : encode_3d(&mq, qkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 3 * C, T, B, pr.hs, BM,
                                   pr.hs == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
  if (!enc) return ATTN_ERR_CUDA;
  // the (B*NH, T, T) fp32 matrices as {T, T, B*NH} for bulk tensor stores of
  // [128][32] chunks; row strides must be multiples of 16 bytes (T % 4 == 0)
  CUtensorMap mp = {}, ma = {};
  const bool tma_out = (T % 4) == 0;
  if (tma_out) {
    auto fn = encode_fn();
    if (!fn) return ATTN_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)T, (cuuint64_t)T, (cuuint64_t)B * NH};
    cuuint64_t strides[2] = {(cuuint64_t)T * 4, (cuuint64_t)T * T * 4};
    cuuint32_t box[3] = {32, 128, 1}, es[3] = {1, 1, 1};
    for (int i = 0; i < 2; ++i) {
      float* base = i == 0 ? preatt : att;
      if (!base) continue;
      if (fn(i == 0 ? &mp : &ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return ATTN_ERR_CUDA;
    }
  }
  cudaError_t ce = launch_att(mq, mp, ma, tma_out, lse, preatt, att, f32, pr, static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

static attn_status_t check_decode(int B, int L, int C, int NH, int Tq, attn_dtype_t dtype) {
  attn_status_t st = check_shape(B, L, C, NH, 1, dtype);
  if (st != ATTN_OK) return st;
  if (Tq < 1 || Tq > L || Tq > decode_max_tq()) return ATTN_ERR_INVALID_ARG;
  const int ch = decode_chunk(dtype == ATTN_F32);
  if ((double)B * NH * ((L + ch - 1) / ch) > 2.0e9) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

extern "C" size_t attn_decode_workspace_size(int B, int L, int C, int NH, int Tq, attn_dtype_t dtype) {
  if (check_decode(B, L, C, NH, Tq, dtype) != ATTN_OK) return 0;
  return decode_workspace_bytes(B, L, C, NH, Tq, dtype == ATTN_F32);
}

extern "C" attn_status_t attn_decode(const void* qkv, void* out, float* lse, int B, int L, int C, int NH, int Tq,
                                     attn_dtype_t dtype, void* workspace, size_t workspace_bytes, void* stream) {
  attn_status_t st = check_decode(B, L, C, NH, Tq, dtype);
  if (st != ATTN_OK) return st;
  if (!qkv || !out || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(out) || !aligned16(lse)) return ATTN_ERR_MISALIGNED;
  const size_t need = decode_workspace_bytes(B, L, C, NH, Tq, dtype == ATTN_F32);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_MISALIGNED;
  const size_t e = esize(dtype);
  const size_t nq = (size_t)B * L * 3 * C * e, no = (size_t)B * Tq * C * e, nl = (size_t)B * NH * Tq * 4;
  if (overlaps(out, no, qkv, nq) || overlaps(lse, nl, qkv, nq) || overlaps(lse, nl, out, no) ||
      overlaps(workspace, need, qkv, nq) || overlaps(workspace, need, out, no) || overlaps(workspace, need, lse, nl))
    return ATTN_ERR_INVALID_ARG;
  if (!device_error_word()) return ATTN_ERR_CUDA;
  const bool f32 = dtype == ATTN_F32;
  CUtensorMap mq, mkq, mqs;
  if (!encode_3d(&mq, qkv, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f32 ? 4 : 2,
                 3 * C, L, B, C / NH, decode_chunk(f32), CU_TENSOR_MAP_SWIZZLE_NONE))
    return ATTN_ERR_CUDA;
  mkq = mq;
  mqs = mq;
  if (!f32) {
    // K and the query rows for the tensor-core scores, in the hs-row swizzle
    const CUtensorMapSwizzle swz = C / NH == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!encode_3d(&mkq, qkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 3 * C, L, B, C / NH, decode_chunk(false), swz) ||
        !encode_3d(&mqs, qkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 3 * C, L, B, C / NH, 16, swz))
      return ATTN_ERR_CUDA;
  }
  cudaError_t ce = launch_decode(mq, mkq, mqs, qkv, out, lse, static_cast<float*>(workspace), f32, B, L, C, NH, Tq,
                                 static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" attn_status_t attn_last_device_error(void* stream) {
  int* addr = device_error_word();
  if (!addr) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, addr, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyAsync(addr, &zero, sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  if (v == 0) return ATTN_OK;
  return (v == ATTN_ERR_TIMEOUT || v == ATTN_ERR_BOUNDS) ? static_cast<attn_status_t>(v) : ATTN_ERR_CUDA;
}

extern "C" attn_status_t attn_profile_enable(int enable) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof.enabled = enable != 0;
  return ATTN_OK;
}

extern "C" attn_status_t attn_profile_reset(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (int k = 0; k < K_COUNT; ++k) {
    if (!profile_drain(k)) return ATTN_ERR_CUDA;
    g_prof.total_ms[k] = 0;
    g_prof.count[k] = 0;
  }
  return ATTN_OK;
}

extern "C" attn_status_t attn_profile_read(int kernel_id, double* total_ms, long long* launches) {
  if (kernel_id < 0 || kernel_id >= K_COUNT || !total_ms || !launches) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!profile_drain(kernel_id)) return ATTN_ERR_CUDA;
  *total_ms = g_prof.total_ms[kernel_id];
  *launches = g_prof.count[kernel_id];
  return ATTN_OK;
}
