// Fused multi-head attention backward for sm_103a (bf16 in, fp32 accumulate)
// on the GPT-2 (B, T, 3C) layout; dqkv is written with = (an activation
// gradient, "llm.c 的中文注解" section 1.1).
//
// Math (llm.c attention_backward_cpu, softmax step in the row-sum form of its
// softmax_autoregressive_backward_kernel7), per (b, h):
//   D_t     = sum_i dout_t[i] out_t[i]            (= sum_j att_tj datt_tj)
//   P_tj    = exp(scale*s_tj - lse_t)              (recomputed from lse)
//   dv_j    = sum_t P_tj dout_t
//   dP_tj   = dout_t . v_j                         (datt)
//   dS_tj   = P_tj (dP_tj - D_t)                   (dpreatt / scale)
//   dk_j    = scale * sum_t dS_tj q_t
//   dq_t    = scale * sum_j dS_tj k_j
//
// Three launches on the caller's stream:
//   1. attn_bwd_pre:    D (fp32, (B,NH,T)) and zero the fp32 dq accumulator (B,T,C)
//   2. attn_bwd_kernel: one CTA per (b, h, 128-key tile), looping over the query
//      tiles that see those keys; S^T, dP^T, dV, dK, dQ on tcgen05, dQ reduced
//      into the accumulator with vector atomics, dK/dV stored with TMA.
//   3. attn_bwd_dq_out: dq accumulator -> bf16 into dqkv[:, :, 0:C].
//
// Main kernel roles (10 warps):
//   warps 0-3  P/dS warpgroup, thread = key row (TMEM lane); dK/dV epilogue
//   warps 4-7  dQ warpgroup, thread = query row; TMEM -> atomics
//   warp  8    loader: K, V once; Q, dO, lse, D per query tile (2 stages)
//   warp  9    MMA issuer
// TMEM columns: S^T [0,128) dP^T [128,256) P^T [256,320) dV [320,384)
//               dK [384,448) dQ [448,512)
#include "common.cuh"

namespace attn {

constexpr int BWD_STAGES = 2;
constexpr int BWD_THREADS = 320;
constexpr uint32_t TB_S = 0, TB_DP = 128, TB_P = 256, TB_DV = 320, TB_DK = 384, TB_DQ = 448;

template <int HS>
struct BwdSmem {
  static constexpr int TILE = TileGeom<HS>::TILE_BYTES;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILE;
  static constexpr int Q_OFF = V_OFF + TILE;                   // BWD_STAGES tiles
  static constexpr int DO_OFF = Q_OFF + BWD_STAGES * TILE;     // BWD_STAGES tiles
  static constexpr int DS_OFF = DO_OFF + BWD_STAGES * TILE;    // dS^T: 2 blocks of [128 keys][64 q]
  static constexpr int DS_BYTES = 2 * 128 * 128;
  static constexpr int ROWST_OFF = DS_OFF + DS_BYTES;          // per stage: lse2[128], D[128]
  static constexpr int BYTES = ROWST_OFF + BWD_STAGES * 2 * 128 * 4;
  static constexpr int ALLOC = BYTES + 1024;
};

struct BwdParams {
  const float* lse;   // (B, NH, T)
  const float* D;     // (B, NH, T)
  float* dq_acc;      // (B, T, C) fp32
  int* err;
  int T, NH, C;
  int n_kv;           // key tiles per head
  int BH;
  float scale;        // 1/sqrt(hs)
  float scale_log2;   // scale * log2(e)
};

// ----------------------------------------------------------------------------
// 1. D = rowsum(dout * out) per head; zero the dq accumulator.
//    One thread per 8 consecutive channels (16 bytes of bf16).
// ----------------------------------------------------------------------------
template <int HS>
__global__ void attn_bwd_pre(const uint4* __restrict__ dout, const uint4* __restrict__ out,
                             float* __restrict__ D, float4* __restrict__ dq_acc, int T, int C, int NH,
                             long long n_vec) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  constexpr int LANES = HS / 8;   // threads per head row
  float acc = 0.f;
  if (i < n_vec) {
    const uint4 a = dout[i], o = out[i];
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      acc = fmaf(__uint_as_float(aw[w] << 16), __uint_as_float(ow[w] << 16), acc);
      acc = fmaf(__uint_as_float(aw[w] & 0xFFFF0000u), __uint_as_float(ow[w] & 0xFFFF0000u), acc);
    }
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    dq_acc[2 * i] = z;
    dq_acc[2 * i + 1] = z;
  }
  // reduce across the LANES threads of one head row (aligned groups in the warp)
#pragma unroll
  for (int off = LANES / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (i < n_vec && (threadIdx.x % LANES) == 0) {
    const long long e = i * 8;                  // element index in (B, T, C)
    const long long bt = e / C;
    const int c = (int)(e - bt * C);
    const int h = c / HS;
    const long long b = bt / T;
    const int t = (int)(bt - b * T);
    D[(b * NH + h) * T + t] = acc;
  }
}

// ----------------------------------------------------------------------------
// 3. dq accumulator (fp32, already scaled) -> bf16 into dqkv[:, :, 0:C].
// ----------------------------------------------------------------------------
__global__ void attn_bwd_dq_out(const float4* __restrict__ dq_acc, uint4* __restrict__ dqkv, int C,
                                long long n_vec) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;   // 8 channels each
  if (i >= n_vec) return;
  const long long e = i * 8;
  const long long bt = e / C;
  const int c = (int)(e - bt * C);
  const float4 a = dq_acc[2 * i], b = dq_acc[2 * i + 1];
  uint4 v;
  v.x = pack_bf16x2(a.x, a.y);
  v.y = pack_bf16x2(a.z, a.w);
  v.z = pack_bf16x2(b.x, b.y);
  v.w = pack_bf16x2(b.z, b.w);
  dqkv[(bt * 3 * C + c) / 8] = v;
}

// ----------------------------------------------------------------------------
// 2. main kernel
// ----------------------------------------------------------------------------
template <int HS, bool CAUSAL>
__global__ void __launch_bounds__(BWD_THREADS, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap map_qkv, const __grid_constant__ CUtensorMap map_dout,
                const __grid_constant__ CUtensorMap map_dqkv, const BwdParams p) {
  using G = TileGeom<HS>;
  using L = BwdSmem<HS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_kv, bar_q_full[BWD_STAGES], bar_q_empty[BWD_STAGES];
  __shared__ uint64_t bar_sdp, bar_p, bar_ds_free, bar_dq_full, bar_dq_free, bar_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kv = (int)(blockIdx.x / p.BH);          // key tile; tile 0 has the most work
  const int bh = blockIdx.x % p.BH;
  const int b = bh / p.NH, h = bh % p.NH;
  const int T = p.T;
  const int n_q_all = (T + BM - 1) / BM;
  const int i0 = CAUSAL ? kv : 0;                   // first query tile that sees these keys
  const int n_it = n_q_all - i0;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < BWD_STAGES; ++s) {
      mbar_init(&bar_q_full[s], 1);
      mbar_init(&bar_q_empty[s], 1);
    }
    mbar_init(&bar_sdp, 1);
    mbar_init(&bar_p, 128);
    mbar_init(&bar_ds_free, 1);
    mbar_init(&bar_dq_full, 1);
    mbar_init(&bar_dq_free, 128);
    mbar_init(&bar_done, 1);
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

  if (warp == 8) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      tma_prefetch_desc(&map_qkv);
      tma_prefetch_desc(&map_dout);
      mbar_arrive_expect_tx(&bar_kv, 2 * G::TILE_BYTES);
      tma_load_3d(smem + L::K_OFF, &map_qkv, &bar_kv, p.C + h * HS, kv * BN, b);
      tma_load_3d(smem + L::V_OFF, &map_qkv, &bar_kv, 2 * p.C + h * HS, kv * BN, b);
    }
    const float log2e = 1.4426950408889634f;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % BWD_STAGES;
      const int qi = i0 + it;
      bool ok = true;
      if (it >= BWD_STAGES) ok = mbar_wait(&bar_q_empty[st], ((it / BWD_STAGES) - 1) & 1, &abort_sh, gerr);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) {
        mbar_expect_tx(&bar_q_full[st], 2 * G::TILE_BYTES);
        tma_load_3d(smem + L::Q_OFF + st * G::TILE_BYTES, &map_qkv, &bar_q_full[st], h * HS, qi * BM, b);
        tma_load_3d(smem + L::DO_OFF + st * G::TILE_BYTES, &map_dout, &bar_q_full[st], h * HS, qi * BM, b);
      }
      float* rs = reinterpret_cast<float*>(smem + L::ROWST_OFF) + st * 256;
      const size_t rowbase = (size_t)bh * T;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int qq = lane + 32 * k;
        const int q = qi * BM + qq;
        // rows past T: lse = +inf makes P = 0 there, D = 0
        rs[qq] = q < T ? p.lse[rowbase + q] * log2e : INFINITY;
        rs[128 + qq] = q < T ? p.D[rowbase + q] : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_q_full[st]);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_sq = make_idesc_bf16(BN, BM, false, false);   // [keys x q], K = HS
      constexpr uint32_t id_kv = make_idesc_bf16(BN, HS, false, true);    // [keys x HS], K = q, B MN-major
      constexpr uint32_t id_dq = make_idesc_bf16(BM, HS, true, true);     // [q x HS], K = keys, A,B MN-major
      const uint32_t sK = smem_u32(smem + L::K_OFF), sV = smem_u32(smem + L::V_OFF);
      const uint32_t sQ = smem_u32(smem + L::Q_OFF), sDO = smem_u32(smem + L::DO_OFF);
      const uint32_t sDS = smem_u32(smem + L::DS_OFF);
      bool ok = mbar_wait(&bar_kv, 0, &abort_sh, gerr);
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it % BWD_STAGES;
        if (!(ok = mbar_wait(&bar_q_full[st], (it / BWD_STAGES) & 1, &abort_sh, gerr))) break;
        tc_fence_after();
        const uint32_t q_a = sQ + st * G::TILE_BYTES, do_a = sDO + st * G::TILE_BYTES;
        // S^T = K Q^T ; dP^T = V dO^T   (K-dim = HS)
#pragma unroll
        for (int k = 0; k < HS / 16; ++k)
          mma_ss(tmem + TB_S, make_sdesc(sK + k * 32, 16, G::ATOM_BYTES, G::SWZ),
                 make_sdesc(q_a + k * 32, 16, G::ATOM_BYTES, G::SWZ), id_sq, k > 0);
#pragma unroll
        for (int k = 0; k < HS / 16; ++k)
          mma_ss(tmem + TB_DP, make_sdesc(sV + k * 32, 16, G::ATOM_BYTES, G::SWZ),
                 make_sdesc(do_a + k * 32, 16, G::ATOM_BYTES, G::SWZ), id_sq, k > 0);
        mma_commit(&bar_sdp);
        if (!(ok = mbar_wait(&bar_p, it & 1, &abort_sh, gerr))) break;
        tc_fence_after();
        // dV += P^T dO  (A = P^T in TMEM, B = dO MN-major; K = 128 queries)
#pragma unroll
        for (int k = 0; k < BM / 16; ++k)
          mma_ts(tmem + TB_DV, tmem + TB_P + k * 8,
                 make_sdesc(do_a + k * 16 * G::ROW_BYTES, 16, G::ATOM_BYTES, G::SWZ), id_kv,
                 (it > 0 || k > 0) ? 1u : 0u);
        // dK += dS^T Q  (A = dS^T K-major: 2 blocks of 64 queries, B = Q MN-major)
#pragma unroll
        for (int k = 0; k < BM / 16; ++k)
          mma_ss(tmem + TB_DK, make_sdesc(sDS + (k / 4) * 16384 + (k % 4) * 32, 16, 1024, SWZ_128B),
                 make_sdesc(q_a + k * 16 * G::ROW_BYTES, 16, G::ATOM_BYTES, G::SWZ), id_kv,
                 (it > 0 || k > 0) ? 1u : 0u);
        if (it > 0) {
          if (!(ok = mbar_wait(&bar_dq_free, (it - 1) & 1, &abort_sh, gerr))) break;
          tc_fence_after();
        }
        // dQ = dS K  (A = dS: MN-major view of the dS^T tile, B = K MN-major; K-dim = 128 keys)
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ss(tmem + TB_DQ, make_sdesc(sDS + k * 16 * 128, 16384, 1024, SWZ_128B),
                 make_sdesc(sK + k * 16 * G::ROW_BYTES, 16, G::ATOM_BYTES, G::SWZ), id_dq, k > 0);
        mma_commit(&bar_dq_full);
        // only commits that someone waits for (no arrival after the CTA retires)
        if (it + 1 < n_it) mma_commit(&bar_ds_free);
        if (it + BWD_STAGES < n_it) mma_commit(&bar_q_empty[st]);
      }
      if (ok) mma_commit(&bar_done);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ P / dS warpgroup
    const int r = (warp << 5) + lane;              // key row in the tile = TMEM lane
    const int key = kv * BN + r;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float c = p.scale_log2;
    bool ok = true;
    uint8_t* sds = smem + L::DS_OFF;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % BWD_STAGES;
      const int qi = i0 + it;
      ok = mbar_wait(&bar_q_full[st], (it / BWD_STAGES) & 1, &abort_sh, gerr);
      ok = ok && mbar_wait(&bar_sdp, it & 1, &abort_sh, gerr);
      if (ok && it > 0) ok = mbar_wait(&bar_ds_free, (it - 1) & 1, &abort_sh, gerr);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* rs = reinterpret_cast<const float*>(smem + L::ROWST_OFF) + st * 256;
      const bool diag = CAUSAL && (qi == kv);
      const bool key_ok = key < T;
#pragma unroll 1
      for (int cq = 0; cq < 4; ++cq) {
        uint32_t sv[32], dpv[32];
        tmem_ld32(tmem + lane_off + TB_S + cq * 32, sv);
        tmem_ld32(tmem + lane_off + TB_DP + cq * 32, dpv);
        tmem_ld_wait(sv);
        tmem_tie32(dpv);
        uint32_t pk[16];
        uint32_t dk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float pp[2], dd[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int qq = cq * 32 + i + u;
            float e = ex2_approx(fmaf(__uint_as_float(sv[i + u]), c, -rs[qq]));
            if (!key_ok || (diag && qq < r)) e = 0.f;
            pp[u] = e;
            dd[u] = e * (__uint_as_float(dpv[i + u]) - rs[128 + qq]);
          }
          pk[i / 2] = pack_bf16x2(pp[0], pp[1]);
          dk[i / 2] = pack_bf16x2(dd[0], dd[1]);
        }
        tmem_st16(tmem + lane_off + TB_P + cq * 16, pk);
        // dS^T row `r`, queries [32cq, 32cq+32): block cq/2, 16-byte chunks 4*(cq%2)..+3
        uint8_t* blk = sds + (cq >> 1) * 16384;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint4 v = make_uint4(dk[ch * 4 + 0], dk[ch * 4 + 1], dk[ch * 4 + 2], dk[ch * 4 + 3]);
          *reinterpret_cast<uint4*>(blk + swz_chunk_offset<64>(r, (cq & 1) * 4 + ch)) = v;
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_p);
    }
    // ---------------------------------------------------------- dK, dV epilogue
    if (ok) {
      ok = mbar_wait(&bar_done, 0, &abort_sh, gerr);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      uint8_t* stage_v = sds;                // dS^T tile is dead after the last MMA
      uint8_t* stage_k = sds + 16384;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? TB_DV : TB_DK;
        const float mul = which == 0 ? 1.f : p.scale;
        uint8_t* stage = which == 0 ? stage_v : stage_k;
#pragma unroll
        for (int cc = 0; cc < HS; cc += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + col + cc, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[ch * 8 + 0]) * mul, __uint_as_float(o[ch * 8 + 1]) * mul);
            v.y = pack_bf16x2(__uint_as_float(o[ch * 8 + 2]) * mul, __uint_as_float(o[ch * 8 + 3]) * mul);
            v.z = pack_bf16x2(__uint_as_float(o[ch * 8 + 4]) * mul, __uint_as_float(o[ch * 8 + 5]) * mul);
            v.w = pack_bf16x2(__uint_as_float(o[ch * 8 + 6]) * mul, __uint_as_float(o[ch * 8 + 7]) * mul);
            *reinterpret_cast<uint4*>(stage + swz_chunk_offset<HS>(r, cc / 8 + ch)) = v;
          }
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (warp == 0 && lane == 0) {
        tma_store_3d(&map_dqkv, stage_v, 2 * p.C + h * HS, kv * BN, b);
        tma_store_3d(&map_dqkv, stage_k, p.C + h * HS, kv * BN, b);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    }
  } else {
    // ------------------------------------------------------------ dQ warpgroup
    const int wq = warp - 4;
    const int r = (wq << 5) + lane;                // query row in the tile
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    for (int it = 0; it < n_it; ++it) {
      const int qi = i0 + it;
      bool ok = mbar_wait(&bar_dq_full, it & 1, &abort_sh, gerr);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t a[HS];
      tmem_ld32(tmem + lane_off + TB_DQ, *reinterpret_cast<uint32_t(*)[32]>(&a[0]));
      if constexpr (HS == 64) tmem_ld32(tmem + lane_off + TB_DQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&a[32]));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&a[0]));
      if constexpr (HS == 64) tmem_tie32(*reinterpret_cast<uint32_t(*)[32]>(&a[32]));
      tc_fence_before();
      mbar_arrive(&bar_dq_free);
      const int t = qi * BM + r;
      if (t < T) {
        float* dst = p.dq_acc + ((size_t)b * T + t) * p.C + h * HS;
        const float s = p.scale;
#pragma unroll
        for (int i = 0; i < HS; i += 4)
          red_add_v4(dst + i, __uint_as_float(a[i]) * s, __uint_as_float(a[i + 1]) * s,
                     __uint_as_float(a[i + 2]) * s, __uint_as_float(a[i + 3]) * s);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (abort_sh) {
    for (int i = 0; i < 1000; ++i) __nanosleep(1000);
  }
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ----------------------------------------------------------------------------
// host launcher
// ----------------------------------------------------------------------------
template <int HS, bool CAUSAL>
static cudaError_t launch_bwd_main(const CUtensorMap& mq, const CUtensorMap& md, const CUtensorMap& mg,
                                   const BwdParams& p, int grid, cudaStream_t stream) {
  auto k = attn_bwd_kernel<HS, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdSmem<HS>::ALLOC);
  if (e != cudaSuccess) return e;
  ProfileScope ps(K_BWD_MAIN, stream);
  k<<<grid, BWD_THREADS, BwdSmem<HS>::ALLOC, stream>>>(mq, md, mg, p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_bf16(const CUtensorMap& map_qkv, const CUtensorMap& map_dout,
                            const CUtensorMap& map_dqkv, const void* dout, const void* out,
                            const float* lse, void* dqkv, float* ws_D, float* ws_dq,
                            const Problem& pr, cudaStream_t stream) {
  const long long n_vec = (long long)pr.B * pr.T * pr.C / 8;
  const int threads = 256;
  const long long blocks = (n_vec + threads - 1) / threads;
  cudaError_t e;
  {
  ProfileScope ps(K_BWD_PRE, stream);
  if (pr.hs == 64)
    attn_bwd_pre<64><<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint4*>(dout), static_cast<const uint4*>(out), ws_D,
        reinterpret_cast<float4*>(ws_dq), pr.T, pr.C, pr.NH, n_vec);
  else
    attn_bwd_pre<32><<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint4*>(dout), static_cast<const uint4*>(out), ws_D,
        reinterpret_cast<float4*>(ws_dq), pr.T, pr.C, pr.NH, n_vec);
  e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;

  BwdParams p;
  p.lse = lse;
  p.D = ws_D;
  p.dq_acc = ws_dq;
  p.err = device_error_word();
  p.T = pr.T;
  p.NH = pr.NH;
  p.C = pr.C;
  p.n_kv = (pr.T + BN - 1) / BN;
  p.BH = pr.B * pr.NH;
  p.scale = (float)(1.0 / __builtin_sqrt((double)pr.hs));
  p.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)pr.hs));
  const int grid = p.n_kv * p.BH;
  if (pr.hs == 64)
    e = pr.causal ? launch_bwd_main<64, true>(map_qkv, map_dout, map_dqkv, p, grid, stream)
                  : launch_bwd_main<64, false>(map_qkv, map_dout, map_dqkv, p, grid, stream);
  else
    e = pr.causal ? launch_bwd_main<32, true>(map_qkv, map_dout, map_dqkv, p, grid, stream)
                  : launch_bwd_main<32, false>(map_qkv, map_dout, map_dqkv, p, grid, stream);
  if (e != cudaSuccess) return e;

  ProfileScope ps(K_BWD_DQ, stream);
  attn_bwd_dq_out<<<(unsigned)blocks, threads, 0, stream>>>(reinterpret_cast<const float4*>(ws_dq),
                                                            static_cast<uint4*>(dqkv), pr.C, n_vec);
  return cudaGetLastError();
}

}  // namespace attn
