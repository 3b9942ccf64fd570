// The linear layers on either side of the attention in the GPT-2 block:
// c_attn (x -> qkv, N = 3C) and c_proj (attention out -> y, N = C), with the
// bias add fused into the GEMM's epilogue, as "LLM Systems 10 & 11:
// Accelerating Transformer Training and Inference" §1.1 (kernel fusion: merge
// the non-GEMM ops of the MHA layer into their neighbours) asks:
//   out[m, o] = bias[o] + sum_k inp[m, k] * weight[o, k]
// inp (M, K) bf16 row-major, weight (N, K) bf16 row-major (llm.c's (OC, C)
// layout), bias (N) bf16 or none, out (M, N) bf16; fp32 accumulation.
//
// Persistent CTAs (one per SM) walk 128 x 256 output tiles. 6 warps:
//   warp 0     TMA producer: A [128][64] and B [256][64] bf16 k-blocks
//              (128-byte swizzle, K-major) through a 4-stage ring
//   warp 1     MMA issuer: tcgen05.mma kind::f16, M = 128, N = 256, K = 16,
//              into one of two TMEM accumulators (256 columns each), so the
//              next tile's MMAs run while this tile's epilogue drains
//   warps 2-5  epilogue: TMEM -> + bias -> bf16 -> a [128][64] staging tile
//              -> TMA store, four 64-column chunks per tile, two staging tiles
// Edges: loads past M, N or K read zeros, stores past M or N are clipped.
#include "../../include/attn.h"
#include "common.cuh"

namespace attn {
namespace lin {

constexpr int TM = 128, TN = 256, TK = 64;
constexpr int ST = 4;
constexpr int THREADS = 192;
constexpr int A_BYTES = TM * TK * 2;      // 16 KB
constexpr int B_BYTES = TN * TK * 2;      // 32 KB
constexpr int STG_BYTES = TM * 64 * 2;    // 16 KB: one 64-column bf16 output chunk
constexpr int A_OFF = 0;
constexpr int B_OFF = A_OFF + ST * A_BYTES;
constexpr int STG_OFF = B_OFF + ST * B_BYTES;
constexpr int SMEM_BYTES = STG_OFF + 2 * STG_BYTES;
constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

struct Params {
  const uint16_t* bias;   // bf16 bits, or null
  int* err;
  int M, N, K;
  int n_n, n_k, n_tiles;
};

__global__ void __launch_bounds__(THREADS, 1)
attn_linear_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_out, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[ST], empty[ST], acc_full[2], acc_empty[2];
  __shared__ float sbias[TN];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_my = p.n_tiles > (int)blockIdx.x ? (p.n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int total_it = n_my * p.n_k;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);            // one arrival per epilogue warp
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  int* gerr = p.err;
  pdl_launch_and_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_a);
      tma_prefetch_desc(&map_b);
      int it = 0;
      bool ok = true;
      for (int lt = 0; ok && lt < n_my; ++lt) {
        const int t = (int)blockIdx.x + lt * (int)gridDim.x;
        const int m0 = (t / p.n_n) * TM, n0 = (t % p.n_n) * TN;
        for (int kb = 0; kb < p.n_k; ++kb, ++it) {
          const int s = it % ST;
          if (it >= ST && !(ok = mbar_wait(&empty[s], ((it / ST) - 1) & 1, &abort_sh, gerr))) break;
          mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
          tma_load_3d(smem + A_OFF + s * A_BYTES, &map_a, &full[s], kb * TK, m0, 0);
          tma_load_3d(smem + B_OFF + s * B_BYTES, &map_b, &full[s], kb * TK, n0, 0);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(TM, TN, false, false);
      const uint64_t dA = make_sdesc(smem_u32(smem + A_OFF), 16, 1024, SWZ_128B);
      const uint64_t dB = make_sdesc(smem_u32(smem + B_OFF), 16, 1024, SWZ_128B);
      int it = 0;
      bool ok = true;
      for (int lt = 0; ok && lt < n_my; ++lt) {
        const int b = lt & 1;
        // the epilogue must have drained this accumulator (tile lt - 2)
        if (lt >= 2 && !(ok = mbar_wait(&acc_empty[b], ((lt >> 1) - 1) & 1, &abort_sh, gerr))) break;
        tc_fence_after();
        for (int kb = 0; kb < p.n_k; ++kb, ++it) {
          const int s = it % ST;
          if (!(ok = mbar_wait(&full[s], (it / ST) & 1, &abort_sh, gerr))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < TK / 16; ++k)
            mma_ss(tmem + b * TN, desc_add(dA, s * A_BYTES + k * 32), desc_add(dB, s * B_BYTES + k * 32), idesc,
                   (kb > 0 || k > 0) ? 1u : 0u);
          // release the stage only if the producer will refill it
          if (it + ST < total_it) mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&acc_full[b]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warpgroup
    const int q = warp & 3;                          // TMEM lane quadrant
    const int r = q * 32 + lane;                     // output row in the tile
    const int et = threadIdx.x - 64;                 // 0..127
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const bool leader = et == 0;
    bool ok = true;
    int chunk = 0;                                   // output chunks stored so far
    for (int lt = 0; ok && lt < n_my; ++lt) {
      const int t = (int)blockIdx.x + lt * (int)gridDim.x;
      const int m0 = (t / p.n_n) * TM, n0 = (t % p.n_n) * TN;
      const int b = lt & 1;
      // bias of this tile's 256 columns (0 past N or without bias)
      for (int c = et; c < TN; c += 128) {
        const int n = n0 + c;
        sbias[c] = (p.bias && n < p.N) ? __uint_as_float((uint32_t)p.bias[n] << 16) : 0.f;
      }
      const bool fail = !mbar_wait(&acc_full[b], (lt >> 1) & 1, &abort_sh, gerr);
      tc_fence_after();
      for (int cc = 0; cc < TN / 64; ++cc, ++chunk) {
        uint8_t* stg = smem + STG_OFF + (chunk & 1) * STG_BYTES;
        // the store issued two chunks ago from this staging tile must have read it
        if (leader) bulk_wait_group_read1();
        if (named_bar_red_or(1, 128, fail)) { ok = false; break; }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + b * TN + cc * 64 + h * 32, v);
          tmem_ld_wait(v);
          const float* bb = sbias + cc * 64 + h * 32;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(v[ch * 8 + 0]) + bb[ch * 8 + 0], __uint_as_float(v[ch * 8 + 1]) + bb[ch * 8 + 1]);
            o.y = pack_bf16x2(__uint_as_float(v[ch * 8 + 2]) + bb[ch * 8 + 2], __uint_as_float(v[ch * 8 + 3]) + bb[ch * 8 + 3]);
            o.z = pack_bf16x2(__uint_as_float(v[ch * 8 + 4]) + bb[ch * 8 + 4], __uint_as_float(v[ch * 8 + 5]) + bb[ch * 8 + 5]);
            o.w = pack_bf16x2(__uint_as_float(v[ch * 8 + 6]) + bb[ch * 8 + 6], __uint_as_float(v[ch * 8 + 7]) + bb[ch * 8 + 7]);
            *reinterpret_cast<uint4*>(stg + swz_chunk_offset<64>(r, h * 4 + ch)) = o;
          }
        }
        if (cc == TN / 64 - 1) {
          // every column of this accumulator is in registers or staged: free it
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && lt + 2 < n_my) mbar_arrive(&acc_empty[b]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          tma_store_3d(&map_out, stg, n0 + cc * 64, m0, 0);
          bulk_commit_group();
        }
      }
      // sbias is rewritten for the next tile only after every thread used it
      named_bar_sync(1, 128);
    }
    if (leader) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (abort_sh) {
    for (int i = 0; i < 1000; ++i) __nanosleep(1000);
  }
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace lin

// map_a: inp {K, M, 1} box {64, 128}; map_b: weight {K, N, 1} box {64, 256};
// map_out: out {N, M, 1} box {64, 128}; all bf16 with the 128-byte swizzle.
cudaError_t launch_linear(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                          const void* bias, int M, int N, int K, cudaStream_t stream) {
  lin::Params p;
  p.bias = static_cast<const uint16_t*>(bias);
  p.err = device_error_word();
  p.M = M;
  p.N = N;
  p.K = K;
  p.n_n = (N + lin::TN - 1) / lin::TN;
  p.n_k = (K + lin::TK - 1) / lin::TK;
  p.n_tiles = ((M + lin::TM - 1) / lin::TM) * p.n_n;
  const int n_sm = device_sm_count();
  const int grid = p.n_tiles < n_sm ? p.n_tiles : n_sm;
  cudaError_t e = cudaFuncSetAttribute(lin::attn_linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       lin::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  ProfileScope ps(K_LINEAR, stream);
  return launch_pdl(lin::attn_linear_kernel, dim3(grid), dim3(lin::THREADS), lin::SMEM_ALLOC, stream, map_a, map_b,
                    map_out, p);
}

}  // namespace attn
