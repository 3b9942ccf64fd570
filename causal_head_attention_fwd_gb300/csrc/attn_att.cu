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
// The work is bound by the HBM writes of the two T x T matrices. Each 128 x 32
// output chunk goes through shared memory: when T % 4 == 0 (16-byte row
// strides) into a 128-byte-swizzled staging tile that one TMA bulk store
// writes out (two tiles alternate, so a store overlaps the next chunk), else
// into a padded tile that the warps store as whole 128-byte row segments.
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
  static constexpr int STG_OFF = 2 * TILE;               // two [128][32] fp32 staging tiles, 128-byte swizzle
  static constexpr int STG_BYTES = 128 * 128;
  static constexpr int ALLOC = STG_OFF + 2 * STG_BYTES + 1024;
};

struct Params {
  const float* lse;
  float* preatt;
  float* att;
  int* err;
  int T, NH, C, BH, n_tiles;
  float scale_log2;
};

template <bool F32, int HS, bool CAUSAL, bool TMA_OUT>
__global__ void __launch_bounds__(THREADS)
attn_att_kernel(const __grid_constant__ CUtensorMap map_qkv, const __grid_constant__ CUtensorMap map_pre,
                const __grid_constant__ CUtensorMap map_att, const Params p) {
  using L = Smem<F32, HS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_ld, bar_mma;
  __shared__ float stage[TMA_OUT ? 1 : BM][33];   // plain-store path: one 128 x 32 fp32 chunk, padded
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
    const bool in = t < T && ATTN_IN_RANGE((size_t)bh * T + t < (size_t)p.BH * T, gerr);
    const float lse2 = in ? p.lse[(size_t)bh * T + t] * 1.4426950408889634f : 0.f;
    const float c = p.scale_log2;
    float* mats[2] = {p.preatt, p.att};
    const CUtensorMap* maps[2] = {&map_pre, &map_att};
    int n = 0;                                   // chunks staged so far (TMA path)
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
        if constexpr (TMA_OUT) {
          // row r's 32 values into a [128][32] fp32 staging tile (128-byte
          // swizzle), then one bulk tensor store; two tiles alternate
          uint8_t* stg = smem + L::STG_OFF + (n & 1) * L::STG_BYTES;
          if (threadIdx.x == 0) bulk_wait_group_read1();   // the store two chunks ago has read this tile
          __syncthreads();
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            float v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int e = ch * 4 + k;
              v[k] = m == 0 ? __uint_as_float(s[e]) : (e < nvis ? ex2_approx(__uint_as_float(s[e]) * c - lse2) : 0.f);
            }
            *reinterpret_cast<float4*>(stg + r * 128 + ((ch ^ (r & 7)) << 4)) = make_float4(v[0], v[1], v[2], v[3]);
          }
          fence_proxy_async_smem();
          __syncthreads();
          if (threadIdx.x == 0) {
            tma_store_3d(maps[m], stg, j0, qt * BM, bh);
            bulk_commit_group();
          }
          ++n;
        } else {
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
            // the last of the four values stays inside the (B, NH, T, T) matrix
            if (!ATTN_IN_RANGE(((size_t)bh * T + tg) * (size_t)T + jg + (jg + 3 < T ? 3 : T - 1 - jg) <
                               (size_t)p.BH * T * (size_t)T, gerr))
              continue;
            float* g = dst + ((size_t)bh * T + tg) * (size_t)T + jg;
#pragma unroll
            for (int x = 0; x < 4; ++x)
              if (jg + x < T) g[x] = stage[rr][c4 + x];
          }
        }
      }
    }
    if constexpr (TMA_OUT) {
      if (threadIdx.x == 0) bulk_wait_group0();   // every store complete before the CTA retires
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

template <bool F32, int HS, bool CAUSAL, bool TMA_OUT>
static cudaError_t launch_t(const CUtensorMap& m, const CUtensorMap& mp, const CUtensorMap& ma, const Params& p,
                            cudaStream_t s) {
  auto k = attn_att_kernel<F32, HS, CAUSAL, TMA_OUT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<F32, HS>::ALLOC);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.BH * p.n_tiles * p.n_tiles;
  k<<<(unsigned)grid, THREADS, Smem<F32, HS>::ALLOC, s>>>(m, mp, ma, p);
  return cudaGetLastError();
}

template <bool F32, int HS>
static cudaError_t launch_hs(const CUtensorMap& m, const CUtensorMap& mp, const CUtensorMap& ma, const Params& p,
                             bool causal, bool tma, cudaStream_t s) {
  if (tma)
    return causal ? launch_t<F32, HS, true, true>(m, mp, ma, p, s) : launch_t<F32, HS, false, true>(m, mp, ma, p, s);
  return causal ? launch_t<F32, HS, true, false>(m, mp, ma, p, s) : launch_t<F32, HS, false, false>(m, mp, ma, p, s);
}

}  // namespace attk

// map_qkv: qkv as {3C, T, B}, box {hs, 128} (bf16) or {32, 128} (fp32);
// map_pre / map_att: the fp32 matrices as {T, T, B*NH}, box {32, 128, 1},
// 128-byte swizzle, used when tma_out (T % 4 == 0) and the matrix is wanted.
cudaError_t launch_att(const CUtensorMap& map_qkv, const CUtensorMap& map_pre, const CUtensorMap& map_att, bool tma_out,
                       const float* lse, float* preatt, float* att, bool f32, const Problem& pr, cudaStream_t stream) {
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
  const bool c = pr.causal != 0;
  if (f32)
    return pr.hs == 64 ? attk::launch_hs<true, 64>(map_qkv, map_pre, map_att, p, c, tma_out, stream)
                       : attk::launch_hs<true, 32>(map_qkv, map_pre, map_att, p, c, tma_out, stream);
  return pr.hs == 64 ? attk::launch_hs<false, 64>(map_qkv, map_pre, map_att, p, c, tma_out, stream)
                     : attk::launch_hs<false, 32>(map_qkv, map_pre, map_att, p, c, tma_out, stream);
}

}  // namespace attn
