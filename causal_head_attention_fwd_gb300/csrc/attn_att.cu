// llm.c drop-in mode: materialise the attention matrices of the forward.
//
// llm.c's attention_forward (dev/cuda/attention_backward.cu) keeps two
// (B, NH, T, T) buffers: preatt = q . k without the scale, the full matrix
// including the masked part, and att = the softmax of scale * preatt over the
// visible keys with the masked entries set to zero (its CPU reference does the
// zeroing "for debugging and checking to PyTorch"). Given qkv and the row
// statistic lse the fused forward wrote, one CTA per (b, h, 128-query tile,
// 128-key tile) computes S = Q K^T on the tensor core (bf16: kind::f16;
// fp32: kind::tf32, both operands K-major straight from the TMA tiles) and
// writes
//   preatt[b,h,t,j] = s_tj                                  (every t, j < T)
//   att[b,h,t,j]    = exp(scale * s_tj - lse_t) if j in J(t), else 0
// The work is bound by the HBM writes of the two T x T matrices; each 128 x 32
// output chunk goes through shared memory so every warp store covers whole
// 128-byte row segments.
#include "../../include/attn.h"
#include "common.cuh"
#include "tf32.cuh"

namespace attn {
namespace attk {

constexpr int THREADS = 128;           // thread = query row of the tile (TMEM lane)

template <bool F32, int HS>
struct Smem {
  // bf16: one [128][HS] tile (128- or 64-byte swizzle); fp32: HS/32 blocks of [128][32]
  static constexpr int TILE = F32 ? HS * 128 * 4 : HS * 128 * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = TILE;
  static constexpr int ALLOC = 2 * TILE + 1024;
};

struct Params {
  const float* lse;
  float* preatt;
  float* att;
  int* err;
  int T, NH, C, BH, n_tiles;
  float scale_log2;
};

template <bool F32, int HS, bool CAUSAL>
__global__ void __launch_bounds__(THREADS)
attn_att_kernel(const __grid_constant__ CUtensorMap map_qkv, const Params p) {
  using L = Smem<F32, HS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_ld, bar_mma;
  __shared__ float stage[BM][33];        // one 128 x 32 fp32 output chunk, padded
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T;
  const int nt = p.n_tiles;
  const int kt = blockIdx.x % nt;
  const int qt = (blockIdx.x / nt) % nt;
  const int bh = blockIdx.x / (nt * nt);
  const int b = bh / p.NH, h = bh % p.NH;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  int* gerr = p.err;

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar_ld, 2 * L::TILE);
    if constexpr (F32) {
#pragma unroll
      for (int c = 0; c < HS / 32; ++c) {
        tma_load_3d(smem + L::Q_OFF + c * 16384, &map_qkv, &bar_ld, h * HS + 32 * c, qt * BM, b);
        tma_load_3d(smem + L::K_OFF + c * 16384, &map_qkv, &bar_ld, p.C + h * HS + 32 * c, kt * BN, b);
      }
    } else {
      tma_load_3d(smem + L::Q_OFF, &map_qkv, &bar_ld, h * HS, qt * BM, b);
      tma_load_3d(smem + L::K_OFF, &map_qkv, &bar_ld, p.C + h * HS, kt * BN, b);
    }
    if (mbar_wait(&bar_ld, 0, &abort_sh, gerr)) {
      tc_fence_after();
      if constexpr (F32) {
        // tf32: K = 8 per MMA (32 bytes of a 128-byte swizzled row); column block kk/4
        constexpr uint32_t idesc = make_idesc_tf32(BM, BN, false, false);
        const uint64_t dq = make_sdesc(smem_u32(smem + L::Q_OFF), 16, 1024, SWZ_128B);
        const uint64_t dk = make_sdesc(smem_u32(smem + L::K_OFF), 16, 1024, SWZ_128B);
#pragma unroll
        for (int kk = 0; kk < HS / 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss_tf32(tmem, desc_add(dq, off), desc_add(dk, off), idesc, kk > 0);
        }
      } else {
        using G = TileGeom<HS>;
        constexpr uint32_t idesc = make_idesc_bf16(BM, BN, false, false);
        const uint64_t dq = make_sdesc(smem_u32(smem + L::Q_OFF), 16, G::ATOM_BYTES, G::SWZ);
        const uint64_t dk = make_sdesc(smem_u32(smem + L::K_OFF), 16, G::ATOM_BYTES, G::SWZ);
#pragma unroll
        for (int k = 0; k < HS / 16; ++k) mma_ss(tmem, desc_add(dq, k * 32), desc_add(dk, k * 32), idesc, k > 0);
      }
      mma_commit(&bar_mma);
    }
  }
  __syncwarp();
  // one decision for the whole CTA: the staged stores below use block barriers
  const bool ok = __syncthreads_and(mbar_wait(&bar_mma, 0, &abort_sh, gerr));
  tc_fence_after();
  const int r = threadIdx.x;
  const int t = qt * BM + r;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  if (ok) {
    const float lse2 = t < T ? p.lse[(size_t)bh * T + t] * 1.4426950408889634f : 0.f;
    const float c = p.scale_log2;
    const bool vec = (T & 3) == 0;             // global rows start 16-byte aligned
    float* mats[2] = {p.preatt, p.att};
#pragma unroll 1
    for (int cc = 0; cc < BN; cc += 32) {
      uint32_t s[32];
      tmem_ld32(tmem + lane_off + cc, s);
      tmem_ld_wait(s);
      const int j0 = kt * BN + cc;
      const int nvis = CAUSAL ? t - j0 + 1 : T - j0;   // keys j0 .. j0+nvis-1 visible
#pragma unroll 1
      for (int m = 0; m < 2; ++m) {
        float* dst = mats[m];
        if (!dst) continue;                        // uniform: the same pointer for every thread
        // thread = row writes its 32 values into a padded [128][33] tile
        // (conflict-free), then each warp stores whole 128-byte row segments
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          stage[r][e] = m == 0 ? __uint_as_float(s[e])
                               : (e < nvis ? ex2_approx(__uint_as_float(s[e]) * c - lse2) : 0.f);
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = k * THREADS + r;           // [128 rows][8 float4] of the chunk
          const int rr = i >> 3, c4 = (i & 7) * 4;
          const int tg = qt * BM + rr, jg = j0 + c4;
          if (tg >= T || jg >= T) continue;
          float* g = dst + ((size_t)bh * T + tg) * (size_t)T + jg;
          if (vec) {
            *reinterpret_cast<float4*>(g) = make_float4(stage[rr][c4], stage[rr][c4 + 1], stage[rr][c4 + 2],
                                                        stage[rr][c4 + 3]);
          } else {
#pragma unroll
            for (int x = 0; x < 4; ++x)
              if (jg + x < T) g[x] = stage[rr][c4 + x];
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

template <bool F32, int HS, bool CAUSAL>
static cudaError_t launch_t(const CUtensorMap& m, const Params& p, cudaStream_t s) {
  auto k = attn_att_kernel<F32, HS, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<F32, HS>::ALLOC);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.BH * p.n_tiles * p.n_tiles;
  k<<<(unsigned)grid, THREADS, Smem<F32, HS>::ALLOC, s>>>(m, p);
  return cudaGetLastError();
}

}  // namespace attk

// map_qkv: qkv as {3C, T, B}, box {hs, 128} (bf16) or {32, 128} (fp32)
cudaError_t launch_att(const CUtensorMap& map_qkv, const float* lse, float* preatt, float* att, bool f32,
                       const Problem& pr, cudaStream_t stream) {
  attk::Params p;
  p.lse = lse;
  p.preatt = preatt;
  p.att = att;
  p.err = device_error_word();
  p.T = pr.T;
  p.NH = pr.NH;
  p.C = pr.C;
  p.BH = pr.B * pr.NH;
  p.n_tiles = (pr.T + BM - 1) / BM;
  p.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)pr.hs));
  if (f32) {
    if (pr.hs == 64)
      return pr.causal ? attk::launch_t<true, 64, true>(map_qkv, p, stream)
                       : attk::launch_t<true, 64, false>(map_qkv, p, stream);
    return pr.causal ? attk::launch_t<true, 32, true>(map_qkv, p, stream)
                     : attk::launch_t<true, 32, false>(map_qkv, p, stream);
  }
  if (pr.hs == 64)
    return pr.causal ? attk::launch_t<false, 64, true>(map_qkv, p, stream)
                     : attk::launch_t<false, 64, false>(map_qkv, p, stream);
  return pr.causal ? attk::launch_t<false, 32, true>(map_qkv, p, stream)
                   : attk::launch_t<false, 32, false>(map_qkv, p, stream);
}

}  // namespace attn
