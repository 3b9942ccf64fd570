// Fused causal / non-causal multi-head attention forward for sm_103a (bf16 in,
// fp32 accumulate), on the GPT-2 (B, T, 3C) qkv layout.
//
// Computes, for every (b, h) and query row t (llm.c attention_forward_cpu,
// passes 1-4; scale = 1/sqrt(hs)):
//   s_tj  = q_t . k_j                       (tcgen05.mma, fp32 in TMEM)
//   p_tj  = exp(scale * (s_tj - m_t)),  j in J(t)   (online, one thread per row)
//   out_t = sum_j p_tj v_j / sum_j p_tj     (tcgen05.mma, fp32 in TMEM)
//   lse_t = scale * m_t + ln sum_j p_tj
// The FlashAttention scheme of "Umakini wa kujitegemea, kerneli za CUDA na
// FlashAttention" section 3: Q/K/V tiles stream through shared memory, the
// T x T score matrix is never written, only out and the row statistic lse.
//
// CTA = two 128-row query tiles of one (b, h) (256 rows), 10 warps:
//   warps 0-3  softmax warpgroup for query tile 0 (TMEM lanes 0-127)
//   warps 4-7  softmax warpgroup for query tile 1
//   warp  8    TMA producer (Q once, then K/V tiles through a 3-stage ring)
//   warp  9    MMA issuer (single thread)
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+HS) O1 [320,320+HS)
//               P0 [384,448) P1 [448,512)  (P = bf16 pairs, 64 columns)
#include "common.cuh"

namespace attn {

constexpr int FWD_STAGES = 3;
constexpr int FWD_THREADS = 320;
constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = 320, TM_P0 = 384, TM_P1 = 448;

template <int HS>
struct FwdSmem {
  static constexpr int TILE = TileGeom<HS>::TILE_BYTES;
  static constexpr int Q_OFF = 0;                          // 2 tiles
  static constexpr int K_OFF = Q_OFF + 2 * TILE;           // FWD_STAGES tiles
  static constexpr int V_OFF = K_OFF + FWD_STAGES * TILE;  // FWD_STAGES tiles
  static constexpr int BYTES = V_OFF + FWD_STAGES * TILE;
  static constexpr int ALLOC = BYTES + 1024;               // room to align to 1024
};

struct FwdParams {
  float* lse;          // (B, NH, T)
  int* err;            // device error word
  int T, NH, C;
  int n_pairs;         // query-tile pairs per head = ceil(T / 256)
  int BH;
  float scale_log2;    // (1/sqrt(hs)) * log2(e)
};

template <int HS, bool CAUSAL>
__global__ void __launch_bounds__(FWD_THREADS, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap map_qkv,
                const __grid_constant__ CUtensorMap map_out, const FwdParams p) {
  using G = TileGeom<HS>;
  using L = FwdSmem<HS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_q, bar_k_full[FWD_STAGES], bar_v_full[FWD_STAGES], bar_kv_empty[FWD_STAGES];
  __shared__ uint64_t bar_s[2], bar_sfree[2], bar_p[2], bar_pv[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: heavy (late) query-tile pairs first so the causal tail is short.
  const int pair = p.n_pairs - 1 - (int)(blockIdx.x / p.BH);
  const int bh = blockIdx.x % p.BH;
  const int b = bh / p.NH, h = bh % p.NH;
  const int T = p.T;
  const int q0 = pair * 2 * BM;               // first query row of tile 0
  const int n_kv_all = (T + BN - 1) / BN;
  int n_tile[2];
  for (int i = 0; i < 2; ++i) {
    const int qs = q0 + i * BM;
    if (qs >= T) n_tile[i] = 0;
    else n_tile[i] = CAUSAL ? (qs / BN + 1) : n_kv_all;
  }
  const int n_max = n_tile[0] > n_tile[1] ? n_tile[0] : n_tile[1];

  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&bar_q, 1);
    for (int s = 0; s < FWD_STAGES; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s[i], 1);
      mbar_init(&bar_sfree[i], 128);
      mbar_init(&bar_p[i], 128);
      mbar_init(&bar_pv[i], 1);
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

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_qkv);
      const uint32_t qbytes = (n_tile[0] > 0 ? G::TILE_BYTES : 0) + (n_tile[1] > 0 ? G::TILE_BYTES : 0);
      mbar_arrive_expect_tx(&bar_q, qbytes);
      for (int i = 0; i < 2; ++i)
        if (n_tile[i] > 0)
          tma_load_3d(smem + L::Q_OFF + i * G::TILE_BYTES, &map_qkv, &bar_q, h * HS, q0 + i * BM, b);
      for (int j = 0; j < n_max; ++j) {
        const int st = j % FWD_STAGES;
        if (j >= FWD_STAGES) {
          if (!mbar_wait(&bar_kv_empty[st], ((j / FWD_STAGES) - 1) & 1, &abort_sh, gerr)) break;
        }
        mbar_arrive_expect_tx(&bar_k_full[st], G::TILE_BYTES);
        tma_load_3d(smem + L::K_OFF + st * G::TILE_BYTES, &map_qkv, &bar_k_full[st], p.C + h * HS, j * BN, b);
        mbar_arrive_expect_tx(&bar_v_full[st], G::TILE_BYTES);
        tma_load_3d(smem + L::V_OFF + st * G::TILE_BYTES, &map_qkv, &bar_v_full[st], 2 * p.C + h * HS, j * BN, b);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc_bf16(BM, BN, false, false);
      constexpr uint32_t idesc_o = make_idesc_bf16(BM, HS, false, true);
      const uint64_t dQ0 = make_sdesc(smem_u32(smem + L::Q_OFF), 16, G::ATOM_BYTES, G::SWZ);
      const uint64_t dK0 = make_sdesc(smem_u32(smem + L::K_OFF), 16, G::ATOM_BYTES, G::SWZ);
      const uint64_t dV0 = make_sdesc(smem_u32(smem + L::V_OFF), 16, G::ATOM_BYTES, G::SWZ);
      // S_i(j) = Q_i K_j^T : K = HS in steps of 16 (32 bytes inside the swizzle row)
      auto issue_s = [&](int i, int st) {
        const uint64_t qd = desc_add(dQ0, i * G::TILE_BYTES), kd = desc_add(dK0, st * G::TILE_BYTES);
        const uint32_t d = tmem + (i ? TM_S1 : TM_S0);
#pragma unroll
        for (int k = 0; k < HS / 16; ++k) mma_ss(d, desc_add(qd, k * 32), desc_add(kd, k * 32), idesc_s, k > 0);
        mma_commit(&bar_s[i]);
      };
      // O_i += P_i V_j : K = 128 keys in steps of 16 (16 rows of V = 2 atoms)
      auto issue_pv = [&](int i, int st, bool acc) {
        const uint64_t vd = desc_add(dV0, st * G::TILE_BYTES);
        const uint32_t d = tmem + (i ? TM_O1 : TM_O0), a = tmem + (i ? TM_P1 : TM_P0);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ts(d, a + k * 8, desc_add(vd, k * 16 * G::ROW_BYTES), idesc_o, (acc || k > 0) ? 1u : 0u);
        mma_commit(&bar_pv[i]);
      };
      bool ok = mbar_wait(&bar_q, 0, &abort_sh, gerr) && mbar_wait(&bar_k_full[0], 0, &abort_sh, gerr);
      if (ok) {
        tc_fence_after();
        for (int i = 0; i < 2; ++i)
          if (n_tile[i] > 0) issue_s(i, 0);
      }
      // Per key tile j: S_i(j+1) for each query tile as soon as its softmax
      // warps hold S_i(j) in registers, then O_i += P_i(j) V_j.
      for (int j = 0; ok && j < n_max; ++j) {
        const int st = j % FWD_STAGES;
        const int st1 = (j + 1) % FWD_STAGES;
        bool k_ready = false;
        for (int i = 0; i < 2 && ok; ++i) {
          if (j + 1 >= n_tile[i]) continue;
          if (!(ok = mbar_wait(&bar_sfree[i], j & 1, &abort_sh, gerr))) break;
          if (!k_ready) {
            if (!(ok = mbar_wait(&bar_k_full[st1], ((j + 1) / FWD_STAGES) & 1, &abort_sh, gerr))) break;
            k_ready = true;
          }
          tc_fence_after();
          issue_s(i, st1);
        }
        if (!ok) break;
        if (!(ok = mbar_wait(&bar_v_full[st], (j / FWD_STAGES) & 1, &abort_sh, gerr))) break;
        for (int i = 0; i < 2 && ok; ++i) {
          if (j >= n_tile[i]) continue;
          if (!(ok = mbar_wait(&bar_p[i], j & 1, &abort_sh, gerr))) break;
          tc_fence_after();
          issue_pv(i, st, j > 0);
        }
        // release the K/V stage only if the producer will refill it (every
        // commit issued is awaited, so no arrival lands after the CTA retires)
        if (ok && j + FWD_STAGES < n_max) mma_commit(&bar_kv_empty[st]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int wg = warp >> 2;                    // query tile index 0/1
    const int r = ((warp & 3) << 5) + lane;      // row inside the tile = TMEM lane
    const int t = q0 + wg * BM + r;              // query row
    const int n = n_tile[wg];
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + (wg ? TM_S1 : TM_S0);
    const uint32_t tO = tmem + lane_off + (wg ? TM_O1 : TM_O0);
    const uint32_t tP = tmem + lane_off + (wg ? TM_P1 : TM_P0);
    const float c = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_s[wg], j & 1, &abort_sh, gerr));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[4][32];
      tmem_ld32(tS + 0, s[0]);
      tmem_ld32(tS + 32, s[1]);
      tmem_ld32(tS + 64, s[2]);
      tmem_ld32(tS + 96, s[3]);
      tmem_ld_wait(s[0]);
      tmem_tie32(s[1]);
      tmem_tie32(s[2]);
      tmem_tie32(s[3]);
      tc_fence_before();
      mbar_arrive(&bar_sfree[wg]);                     // S columns may be overwritten now
      // mask: causal diagonal tile (key > row), or keys past T (non-causal tail)
      const int kbase = j * BN;
      int limit = BN;                                  // keys [kbase, kbase+limit) are visible
      if (CAUSAL) { if (kbase + BN > t) limit = t - kbase + 1; }
      else { if (kbase + BN > T) limit = T - kbase; }
      if (__any_sync(0xffffffffu, limit < BN)) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (q * 32 + i >= limit) s[q][i] = __float_as_uint(-INFINITY);
      }
      // row max: 3-input max in 8 independent chains, then a short tree
      float mx8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          mx8[(i >> 1) & 7] = fmax3(mx8[(i >> 1) & 7], __uint_as_float(s[q][i]), __uint_as_float(s[q][i + 1]));
      const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
      // Lazy rescaling: the exponent reference m_run only moves when the row
      // max exceeds it by more than 8 (log2 units), so p <= 2^8 and O is
      // rescaled rarely. Result and lse are exact for any reference value.
      const float m_new = (mx - m_run) * c > 8.f ? mx : m_run;
      const float alpha = ex2_approx((m_run - m_new) * c);
      const float2 c2 = make_float2(c, c), nmc = make_float2(-m_new * c, -m_new * c);
      float2 ls[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
      // p = exp2(s*c - m*c) in packed pairs; P goes to TMEM in two 64-key halves
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pk[32];
#pragma unroll
        for (int qq = 0; qq < 2; ++qq)
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const int q = hf * 2 + qq;
            const float2 x = fma2(make_float2(__uint_as_float(s[q][i]), __uint_as_float(s[q][i + 1])), c2, nmc);
            const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            ls[(i >> 1) & 3] = add2(ls[(i >> 1) & 3], e);
            pk[qq * 16 + i / 2] = pack_bf16x2(e.x, e.y);
          }
        if (hf == 0 && j > 0) {
          // P_{j-1} must have been consumed (and O updated) by the previous P.V
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_pv[wg], (j - 1) & 1, &abort_sh, gerr));
          if (!ok) break;
          tc_fence_after();
          // rescale the running output when this row's reference max moved
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int cc = 0; cc < HS; cc += 32) {
              uint32_t o[32];
              tmem_ld32(tO + cc, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(tO + cc, o);
            }
          }
        }
        tmem_st32(tP + hf * 32, pk);
      }
      if (!ok) break;
      const float lsum = ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
      l_run = l_run * alpha + lsum;
      m_run = m_new;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_p[wg]);
    }
    // ---------------------------------------------------------- epilogue
    if (n > 0 && ok) {
      ok = mbar_wait(&bar_pv[wg], (n - 1) & 1, &abort_sh, gerr);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (n > 0 && ok) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      uint8_t* stage = smem + L::Q_OFF + wg * G::TILE_BYTES;   // Q tile is dead now
#pragma unroll
      for (int cc = 0; cc < HS; cc += 32) {
        uint32_t o[32];
        tmem_ld32(tO + cc, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {         // four 16-byte chunks = 32 values
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(o[ch * 8 + 0]) * inv_l, __uint_as_float(o[ch * 8 + 1]) * inv_l);
          v.y = pack_bf16x2(__uint_as_float(o[ch * 8 + 2]) * inv_l, __uint_as_float(o[ch * 8 + 3]) * inv_l);
          v.z = pack_bf16x2(__uint_as_float(o[ch * 8 + 4]) * inv_l, __uint_as_float(o[ch * 8 + 5]) * inv_l);
          v.w = pack_bf16x2(__uint_as_float(o[ch * 8 + 6]) * inv_l, __uint_as_float(o[ch * 8 + 7]) * inv_l);
          *reinterpret_cast<uint4*>(stage + swz_chunk_offset<HS>(r, cc / 8 + ch)) = v;
        }
      }
      if (t < T) {
        // lse = scale*m + ln(l) = (m*c + log2 l) * ln 2
        p.lse[(size_t)(b * p.NH + h) * T + t] = (m_run * c + __log2f(l_run)) * 0.69314718055994531f;
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + wg, 128);
      if ((warp & 3) == 0 && lane == 0) {
        tma_store_3d(&map_out, stage, h * HS, q0 + wg * BM, b);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (abort_sh) {
    // give copies already in flight time to land before the CTA retires
    for (int i = 0; i < 1000; ++i) __nanosleep(1000);
  }
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ----------------------------------------------------------------------------
// host launcher
// ----------------------------------------------------------------------------
template <int HS, bool CAUSAL>
static cudaError_t launch_fwd_t(const CUtensorMap& mq, const CUtensorMap& mo, const FwdParams& p,
                                int grid, cudaStream_t stream) {
  auto k = attn_fwd_kernel<HS, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdSmem<HS>::ALLOC);
  if (e != cudaSuccess) return e;
  ProfileScope ps(K_FWD, stream);
  k<<<grid, FWD_THREADS, FwdSmem<HS>::ALLOC, stream>>>(mq, mo, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_bf16(const CUtensorMap& map_qkv, const CUtensorMap& map_out, float* lse,
                            const Problem& pr, cudaStream_t stream) {
  FwdParams p;
  p.lse = lse;
  p.err = device_error_word();
  p.T = pr.T;
  p.NH = pr.NH;
  p.C = pr.C;
  p.n_pairs = (pr.T + 2 * BM - 1) / (2 * BM);
  p.BH = pr.B * pr.NH;
  p.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)pr.hs));
  const int grid = p.n_pairs * p.BH;
  if (pr.hs == 64)
    return pr.causal ? launch_fwd_t<64, true>(map_qkv, map_out, p, grid, stream)
                     : launch_fwd_t<64, false>(map_qkv, map_out, p, grid, stream);
  return pr.causal ? launch_fwd_t<32, true>(map_qkv, map_out, p, grid, stream)
                   : launch_fwd_t<32, false>(map_qkv, map_out, p, grid, stream);
}

}  // namespace attn
