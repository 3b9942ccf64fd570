// Shared definitions of the attention kernels and their host launchers.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace attn {

constexpr int BM = 128;   // query rows per tile (TMEM lanes)
constexpr int BN = 128;   // keys per tile

// Swizzle geometry of a [rows][HS] bf16 tile: HS=64 -> 128-byte rows (SW128),
// HS=32 -> 64-byte rows (SW64). One swizzle atom is 8 rows.
template <int HS>
struct TileGeom {
  static constexpr int ROW_BYTES = HS * 2;
  static constexpr int ATOM_BYTES = 8 * ROW_BYTES;
  static constexpr uint32_t SWZ = (HS == 64) ? SWZ_128B : SWZ_64B;
  static constexpr int TILE_BYTES = BM * ROW_BYTES;   // 128 rows
  static_assert(HS == 32 || HS == 64, "head size must be 32 or 64");
};

// Byte offset of the 16-byte chunk `c` of row `r` inside a swizzled tile.
template <int HS>
__device__ __forceinline__ uint32_t swz_chunk_offset(int r, int c) {
  if constexpr (HS == 64) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
  } else {
    return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
  }
}

// Host-side view of one call (already validated).
struct Problem {
  int B, T, C, NH, hs, causal;
};

// Device address of the library's error word (0 = fine, otherwise an
// attn_status_t code written by a kernel whose bounded wait gave up).
int* device_error_word();

// Process-unique id of the current CUDA context (false if none is current).
bool current_context_id(unsigned long long* id);

// Number of SMs of the current device (cached; persistent grids are sized by it).
int device_sm_count();

// Optional per-kernel timing (see attn_profile_enable in include/attn.h).
enum KernelId { K_FWD = 0, K_BWD_PRE = 1, K_BWD_MAIN = 2, K_BWD_DQ = 3, K_LINEAR = 4, K_COUNT = 5 };
void profile_begin(KernelId k, cudaStream_t s);
void profile_end(KernelId k, cudaStream_t s);

struct ProfileScope {
  KernelId k;
  cudaStream_t s;
  ProfileScope(KernelId k_, cudaStream_t s_) : k(k_), s(s_) { profile_begin(k, s); }
  ~ProfileScope() { profile_end(k, s); }
};

// Launch `k` with programmatic stream serialization: it may start launching
// while the previous kernel on `s` finishes; the kernel itself waits
// (pdl_launch_and_wait) before it touches memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace attn
