// Causal / non-causal multi-head attention, forward and backward, for fp32
// inputs on sm_103a, on the GPT-2 (B, T, 3C) qkv layout. The contractions run
// on the tensor core as tcgen05.mma kind::tf32 with fp32 accumulation in TMEM;
// the FlashAttention scheme of "Umakini wa kujitegemea, kerneli za CUDA na
// FlashAttention" section 3 (tiles through shared memory, no T x T matrix,
// P recomputed from lse in the backward).
//
// What is computed is the same as for bf16 inputs (llm.c attention_forward_cpu
// and attention_backward_cpu, with the softmax backward in the row-sum form of
// its softmax_autoregressive_backward_kernel7; scale = 1/sqrt(hs)).
//
// fp32 tiles are twice the size of bf16 ones, so the kernels stream 64-row
// tiles against a fixed 128-row tile:
//   attn_fwd_f32_kernel   CTA = two 128-row query tiles; 64-key steps, the
//                         score buffer double-buffered in TMEM and P written
//                         over S in place (TS form for O += P V)
//   attn_bwd_pre_f32      D = rowsum(dO * O)
//   attn_bwd_dkdv_f32     CTA = one 128-key tile; walks 64-row query tiles:
//                         S^T = K Q^T, dP^T = V dO^T, P^T and dS^T written over
//                         them in TMEM, dV += P^T dO and dK += dS^T Q (TS)
//   attn_bwd_dq_f32       CTA = one 128-row query tile; walks 64-key tiles:
//                         S = Q K^T, dP = dO V^T, dS over dP, dQ += dS K (TS);
//                         dQ goes to dqkv with a plain store (no atomics)
// Shared-memory tiles: [rows][hs] fp32 split into hs/32 column blocks of
// [rows][32] (128-byte rows, 128-byte swizzle), as the TMA writes them.
// With tf32 operands the tensor core takes shared-memory operands K-major
// only (an MN-major tf32 operand yields zeros on this GPU), so the operand
// whose contraction index runs along its rows (V for P V; Q, dO for dK, dV;
// K for dQ) is transposed in shared memory by two transposer warps per CTA
// into [hs rows][64] K-major tiles, rounding to tf32 on the way.
// Values the kernels produce for the tensor core (P, dS) are rounded to tf32
// too; Q, K, dO read straight from the TMA tiles (for Q K^T, dO V^T) are used
// as stored (the tensor core ignores their 13 low mantissa bits).
#include "common.cuh"
#include "tf32.cuh"

namespace attn {
namespace f32k {

constexpr int BQ = 128;        // rows of a fixed tile (TMEM lanes)
constexpr int BS = 64;         // rows of a streamed tile (one step)
constexpr float LOG2E = 1.4426950408889634f;

template <int HS>
struct Geom {
  static_assert(HS == 32 || HS == 64, "head size must be 32 or 64");
  static constexpr int NB = HS / 32;          // 128-byte column blocks per row
  static constexpr int BLK_L = BQ * 128;      // one block of a 128-row tile (16 KB)
  static constexpr int BLK_S = BS * 128;      // one block of a 64-row tile (8 KB)
  static constexpr int TILE_L = NB * BLK_L;
  static constexpr int TILE_S = NB * BLK_S;
};

// Byte offset of the 16-byte chunk `ch` (0..7) of row r in a 128-byte-swizzled block.
__device__ __forceinline__ uint32_t sw128(int r, int ch) {
  return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4));
}

// K-major operand, MMA step kk (8 tf32 = 32 bytes of K): column block kk/4,
// 32-byte offset inside the swizzled row.
template <int BLK>
__device__ __forceinline__ uint32_t kmaj_step(int kk) {
  return (uint32_t)((kk >> 2) * BLK + (kk & 3) * 32);
}

// TMA load of a [ROWS][HS] fp32 tile as HS/32 column blocks.
template <int HS, int ROWS>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int x0, int y0,
                                          int z) {
#pragma unroll
  for (int c = 0; c < HS / 32; ++c) tma_load_3d(dst + c * ROWS * 128, m, bar, x0 + 32 * c, y0, z);
}

// TMA store of a staged [128][HS] fp32 tile.
template <int HS>
__device__ __forceinline__ void store_tile(const CUtensorMap* m, const uint8_t* src, int x0, int y0, int z) {
#pragma unroll
  for (int c = 0; c < HS / 32; ++c) tma_store_3d(m, src + c * BQ * 128, x0 + 32 * c, y0, z);
}

// Write 32 fp32 values (columns cc..cc+31 of row r, times `mul`) into a staged
// [128][HS] tile.
__device__ __forceinline__ void stage32(uint8_t* tile, int r, int cc, const uint32_t (&v)[32], float mul) {
  uint8_t* blk = tile + (cc >> 5) * (BQ * 128);
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    const float4 f = make_float4(__uint_as_float(v[4 * ch + 0]) * mul, __uint_as_float(v[4 * ch + 1]) * mul,
                                 __uint_as_float(v[4 * ch + 2]) * mul, __uint_as_float(v[4 * ch + 3]) * mul);
    *reinterpret_cast<float4*>(blk + sw128(r, ch)) = f;
  }
}

// Load 64 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[2][32]) {
  tmem_ld32(taddr, r[0]);
  tmem_ld32(taddr + 32, r[1]);
  tmem_ld_wait(r[0]);
  tmem_tie32(r[1]);
}

constexpr int NT = 2;                 // transposer warps per CTA

// One 32x32 sub-block `sb` of the transpose of a streamed [64 rows][HS] tile
// (HS/32 blocks of [64][32]) into [HS rows][64] (2 blocks of [HS][32]), both
// with the 128-byte swizzle; values rounded to tf32. Sub-block sb covers
// source rows 32*(sb&1).. and source columns 32*(sb>>1)..; lane = source row.
// Reads: each lane one 16-byte chunk of its row (conflict-free under the
// swizzle); writes: for each destination row the 32 lanes fill 32 consecutive
// words (conflict-free).
template <int HS>
__device__ __forceinline__ void transpose_sub(const uint8_t* src, uint8_t* dst, int sb, int lane) {
  const int rb = sb & 1, cb = sb >> 1;
  const int row = 32 * rb + lane;
  const uint8_t* s = src + cb * (BS * 128);
  uint8_t* d = dst + rb * (HS * 128);
  const uint32_t col = (uint32_t)(lane & 3) * 4;
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    const float4 v = *reinterpret_cast<const float4*>(s + sw128(row, ch));
    const int r0 = 32 * cb + 4 * ch;
    *reinterpret_cast<uint32_t*>(d + sw128(r0 + 0, lane >> 2) + col) = round_tf32(v.x);
    *reinterpret_cast<uint32_t*>(d + sw128(r0 + 1, lane >> 2) + col) = round_tf32(v.y);
    *reinterpret_cast<uint32_t*>(d + sw128(r0 + 2, lane >> 2) + col) = round_tf32(v.z);
    *reinterpret_cast<uint32_t*>(d + sw128(r0 + 3, lane >> 2) + col) = round_tf32(v.w);
  }
}

// ============================================================================
// forward
// ============================================================================
// TMEM columns of query tile i (base 256*i): S buffers [0,64) and [64,128)
// (P overwrites S in place), O [128, 128+HS).
// Warps: 0-3 / 4-7 softmax of query tile 0 / 1, 8 TMA producer, 9 MMA issuer,
// 10-11 V transposers.
constexpr int FWD_THREADS = 384;
constexpr int FWD_STAGES = 3;     // K / V ring
constexpr int FWD_TSTAGES = 2;    // transposed V ring

template <int HS>
struct FwdSmem {
  using G = Geom<HS>;
  static constexpr int Q_OFF = 0;                                   // 2 tiles of 128 rows
  static constexpr int K_OFF = Q_OFF + 2 * G::TILE_L;               // FWD_STAGES tiles of 64 rows
  static constexpr int V_OFF = K_OFF + FWD_STAGES * G::TILE_S;
  static constexpr int VT_OFF = V_OFF + FWD_STAGES * G::TILE_S;     // FWD_TSTAGES [HS][64] tiles
  static constexpr int BYTES = VT_OFF + FWD_TSTAGES * G::TILE_S;
  static constexpr int ALLOC = BYTES + 1024;
};

struct FwdParams {
  float* lse;
  int* err;
  int T, NH, C, BH, n_pairs;
  float scale_log2;
};

template <int HS, bool CAUSAL>
__global__ void __launch_bounds__(FWD_THREADS, 1)
attn_fwd_f32_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv,
                    const __grid_constant__ CUtensorMap map_out, const FwdParams p) {
  using G = Geom<HS>;
  using L = FwdSmem<HS>;
  constexpr int ST = FWD_STAGES, ST2 = FWD_TSTAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_q, bar_k_full[ST], bar_v_full[ST], bar_kv_empty[ST];
  __shared__ uint64_t bar_vt_full[ST2], bar_vt_empty[ST2];
  __shared__ uint64_t bar_s[2][2], bar_p[2], bar_pv[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = p.T;
  const int pair = p.n_pairs - 1 - (int)(blockIdx.x / p.BH);   // long causal rows first
  const int bh = blockIdx.x % p.BH;
  const int b = bh / p.NH, h = bh % p.NH;
  const int q0 = pair * 2 * BQ;
  const int n_all = (T + BS - 1) / BS;
  int n_tile[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int qs = q0 + i * BQ;
    const int kend = CAUSAL ? min(qs + BQ, T) : T;
    n_tile[i] = qs >= T ? 0 : (CAUSAL ? (kend + BS - 1) / BS : n_all);
  }
  const int n_max = max(n_tile[0], n_tile[1]);

  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&bar_q, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1 + NT);           // K by the MMAs, V by the transposer warps
    }
    for (int s = 0; s < ST2; ++s) {
      mbar_init(&bar_vt_full[s], NT);
      mbar_init(&bar_vt_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s[i][0], 1);
      mbar_init(&bar_s[i][1], 1);
      mbar_init(&bar_p[i], 4);                  // one arrival per softmax warp
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
      const uint32_t qbytes = (n_tile[0] > 0 ? G::TILE_L : 0) + (n_tile[1] > 0 ? G::TILE_L : 0);
      mbar_arrive_expect_tx(&bar_q, qbytes);
      for (int i = 0; i < 2; ++i)
        if (n_tile[i] > 0)
          load_tile<HS, BQ>(smem + L::Q_OFF + i * G::TILE_L, &map_q, &bar_q, h * HS, q0 + i * BQ, b);
      for (int j = 0; j < n_max; ++j) {
        const int st = j % ST;
        if (j >= ST && !mbar_wait(&bar_kv_empty[st], ((j / ST) - 1) & 1, &abort_sh, gerr)) break;
        mbar_arrive_expect_tx(&bar_k_full[st], G::TILE_S);
        load_tile<HS, BS>(smem + L::K_OFF + st * G::TILE_S, &map_kv, &bar_k_full[st], p.C + h * HS, j * BS, b);
        mbar_arrive_expect_tx(&bar_v_full[st], G::TILE_S);
        load_tile<HS, BS>(smem + L::V_OFF + st * G::TILE_S, &map_kv, &bar_v_full[st], 2 * p.C + h * HS, j * BS,
                          b);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc_tf32(BQ, BS, false, false);
      constexpr uint32_t idesc_o = make_idesc_tf32(BQ, HS, false, false);
      const uint64_t dQ0 = make_sdesc(smem_u32(smem + L::Q_OFF), 16, 1024, SWZ_128B);
      const uint64_t dK0 = make_sdesc(smem_u32(smem + L::K_OFF), 16, 1024, SWZ_128B);
      const uint64_t dVT0 = make_sdesc(smem_u32(smem + L::VT_OFF), 16, 1024, SWZ_128B);
      auto issue_s = [&](int i, int j) {
        const uint64_t qd = desc_add(dQ0, i * G::TILE_L), kd = desc_add(dK0, (j % ST) * G::TILE_S);
        const uint32_t d = tmem + i * 256 + (j & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < HS / 8; ++kk)
          mma_ss_tf32(d, desc_add(qd, kmaj_step<G::BLK_L>(kk)), desc_add(kd, kmaj_step<G::BLK_S>(kk)), idesc_s,
                      kk > 0);
        mma_commit(&bar_s[i][j & 1]);
      };
      // O_i += P_i(j) V_j: A = P from TMEM, B = V^T [HS][64 keys] K-major
      auto issue_pv = [&](int i, int j) {
        const uint64_t vd = desc_add(dVT0, (j % ST2) * G::TILE_S);
        const uint32_t d = tmem + i * 256 + 128, a = tmem + i * 256 + (j & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < BS / 8; ++kk)
          mma_ts_tf32(d, a + kk * 8, desc_add(vd, kmaj_step<HS * 128>(kk)), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar_pv[i]);
      };
      auto scores = [&](int j) -> bool {        // S_i(j) of both tiles; releases K_j when they finish
        if (!mbar_wait(&bar_k_full[j % ST], (j / ST) & 1, &abort_sh, gerr)) return false;
        for (int i = 0; i < 2; ++i) {
          if (j >= n_tile[i]) continue;
          // S(j) overwrites the buffer P(j-2) sat in: O += P(j-2) V must be done
          if (j >= 2 && !mbar_wait(&bar_pv[i], (j - 2) & 1, &abort_sh, gerr)) return false;
          tc_fence_after();
          issue_s(i, j);
        }
        if (j + ST < n_max) mma_commit(&bar_kv_empty[j % ST]);
        return true;
      };
      bool ok = mbar_wait(&bar_q, 0, &abort_sh, gerr);
      for (int jj = 0; ok && jj < 2 && jj < n_max; ++jj) ok = scores(jj);
      for (int j = 0; ok && j < n_max; ++j) {
        const int st2 = j % ST2;
        if (!(ok = mbar_wait(&bar_vt_full[st2], (j / ST2) & 1, &abort_sh, gerr))) break;
        for (int i = 0; i < 2 && ok; ++i) {
          if (j >= n_tile[i]) continue;
          if (!(ok = mbar_wait(&bar_p[i], j & 1, &abort_sh, gerr))) break;
          tc_fence_after();
          issue_pv(i, j);
        }
        if (!ok) break;
        if (j + ST2 < n_max) mma_commit(&bar_vt_empty[st2]);
        if (j + 2 < n_max) ok = scores(j + 2);
      }
    }
  } else if (warp >= 10) {
    // ------------------------------------------------------------ V transposers
    const int wt = warp - 10;
    bool ok = true;
    for (int j = 0; ok && j < n_max; ++j) {
      const int st = j % ST, st2 = j % ST2;
      ok = mbar_wait(&bar_v_full[st], (j / ST) & 1, &abort_sh, gerr);
      if (ok && j >= ST2) ok = mbar_wait(&bar_vt_empty[st2], ((j / ST2) - 1) & 1, &abort_sh, gerr);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      for (int sb = wt; sb < 2 * G::NB; sb += NT)
        transpose_sub<HS>(smem + L::V_OFF + st * G::TILE_S, smem + L::VT_OFF + st2 * G::TILE_S, sb, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar_vt_full[st2]);
        if (j + ST < n_max) mbar_arrive(&bar_kv_empty[st]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int wg = warp >> 2;
    const int r = ((warp & 3) << 5) + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tbase = tmem + lane_off + wg * 256;
    const uint32_t tO = tbase + 128;
    const bool leader = (warp & 3) == 0 && lane == 0;
    const float c = p.scale_log2;
    const int n = n_tile[wg];
    const int t = q0 + wg * BQ + r;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const uint32_t tS = tbase + (j & 1) * 64;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_s[wg][j & 1], (j >> 1) & 1, &abort_sh, gerr));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[2][32];
      tmem_ld64(tS, s);
      const int kbase = j * BS;
      const int limit = CAUSAL ? t - kbase + 1 : T - kbase;   // keys [kbase, kbase+limit) visible
      if (__any_sync(0xffffffffu, limit < BS)) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (q * 32 + e >= limit) s[q][e] = __float_as_uint(-INFINITY);
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          mx4[(e >> 1) & 3] = fmax3(mx4[(e >> 1) & 3], __uint_as_float(s[q][e]), __uint_as_float(s[q][e + 1]));
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      // lazy rescaling as in the bf16 forward: the reference only moves when
      // the row max exceeds it by more than 8 (log2 units)
      const float m_new = (mx - m_run) * c > 8.f ? mx : m_run;
      const float alpha = ex2_approx((m_run - m_new) * c);
      const float2 c2 = make_float2(c, c), nmc = make_float2(-m_new * c, -m_new * c);
      float2 ls[2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 x = fma2(make_float2(__uint_as_float(s[q][e]), __uint_as_float(s[q][e + 1])), c2, nmc);
          const float2 ev = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          ls[(e >> 1) & 1] = add2(ls[(e >> 1) & 1], ev);
          s[q][e] = round_tf32(ev.x);
          s[q][e + 1] = round_tf32(ev.y);
        }
      if (j > 0) {
        // O += P(j-1) V must be complete before O is rescaled
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_pv[wg], (j - 1) & 1, &abort_sh, gerr));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int cc = 0; cc < HS; cc += 32) {
            uint32_t o[32];
            tmem_ld32(tO + cc, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + cc, o);
          }
        }
      }
      tmem_st32(tS, s[0]);
      tmem_st32(tS + 32, s[1]);
      l_run = l_run * alpha + ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y));
      m_run = m_new;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p[wg]);
    }
    // every thread of the warpgroup takes the same branch at the barriers below
    ok = !named_bar_red_or(1 + wg, 128, !ok);
    if (ok && n > 0) {
      uint8_t* stage = smem + L::Q_OFF + wg * G::TILE_L;     // this Q tile is dead now
      const bool fail = !mbar_wait(&bar_pv[wg], (n - 1) & 1, &abort_sh, gerr);
      tc_fence_after();
      const float inv_l = 1.f / l_run;
#pragma unroll
      for (int cc = 0; cc < HS; cc += 32) {
        uint32_t o[32];
        tmem_ld32(tO + cc, o);
        tmem_ld_wait(o);
        stage32(stage, r, cc, o, inv_l);
      }
      if (t < T && !fail && ATTN_IN_RANGE((size_t)bh * T + t < (size_t)p.BH * T, gerr))
        p.lse[(size_t)bh * T + t] = (m_run * c + __log2f(l_run)) * 0.69314718055994531f;
      fence_proxy_async_smem();
      if (!named_bar_red_or(1 + wg, 128, fail) && leader) {
        store_tile<HS>(&map_out, stage, h * HS, q0 + wg * BQ, b);
        bulk_commit_group();
        bulk_wait_group_read0();
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

// ============================================================================
// backward: D pre-pass
// ============================================================================
// D[b,h,t] = sum_i dout[b,t,h*hs+i] * out[b,t,h*hs+i]; one thread per 4 channels,
// HS/4 threads per head row reduce with shuffles.
template <int HS>
__global__ void __launch_bounds__(256)
attn_bwd_pre_f32(const float* __restrict__ dout, const float* __restrict__ out, float* __restrict__ D, int T,
                 int C, int NH, long long n_threads, int* err) {
  constexpr int LANES = HS / 4;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const bool valid = i < n_threads;
  const long long ii = valid ? i : 0;
  const long long row = ii / (C / 4);               // b*T + t
  const int ch = (int)(ii % (C / 4)) * 4;
  float s = 0.f;
  if (valid) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(dout + row * C + ch));
    const float4 o = __ldg(reinterpret_cast<const float4*>(out + row * C + ch));
    s = (a.x * o.x + a.y * o.y) + (a.z * o.z + a.w * o.w);
  }
#pragma unroll
  for (int off = LANES / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (valid && (ch % HS) == 0) {
    const long long bb = row / T, t = row % T;
    const long long di = (bb * NH + ch / HS) * T + t;
    if (ATTN_IN_RANGE(di < n_threads * 4 / C * NH, err)) D[di] = s;   // D has B*T*NH entries
  }
}

// ============================================================================
// backward: dK, dV (one CTA per 128-key tile)
// ============================================================================
// TMEM: S^T buffers [0,64) [64,128) (P^T in place), dP^T buffers [128,192)
// [192,256) (dS^T in place), dV [256, 256+HS), dK [320, 320+HS).
// Warps: 0-3 P^T/dS^T (thread = key row), 4 TMA loader, 5 MMA issuer,
// 6-7 Q/dO transposers.
constexpr int BWD_THREADS = 256;
constexpr int DKDV_STAGES = 2;    // Q / dO ring
constexpr int DKDV_TSTAGES = 2;   // transposed Q / dO ring

template <int HS>
struct DkdvSmem {
  using G = Geom<HS>;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + G::TILE_L;
  static constexpr int Q_OFF = V_OFF + G::TILE_L;                   // DKDV_STAGES tiles of 64 rows
  static constexpr int DO_OFF = Q_OFF + DKDV_STAGES * G::TILE_S;
  static constexpr int QT_OFF = DO_OFF + DKDV_STAGES * G::TILE_S;   // DKDV_TSTAGES [HS][64] tiles
  static constexpr int DOT_OFF = QT_OFF + DKDV_TSTAGES * G::TILE_S;
  static constexpr int ROW_OFF = DOT_OFF + DKDV_TSTAGES * G::TILE_S; // [2][lse*log2e 64, D 64]
  static constexpr int BYTES = ROW_OFF + 2 * 128 * 4;
  static constexpr int ALLOC = BYTES + 1024;
};

struct BwdParams {
  const float* lse;
  const float* D;
  int* err;
  int T, NH, C, BH, n_tiles;
  float scale, scale_log2;
};

template <int HS, bool CAUSAL>
__global__ void __launch_bounds__(BWD_THREADS, 1)
attn_bwd_dkdv_f32(const __grid_constant__ CUtensorMap map_kv, const __grid_constant__ CUtensorMap map_qs,
                  const __grid_constant__ CUtensorMap map_dos, const __grid_constant__ CUtensorMap map_g,
                  const BwdParams p) {
  using G = Geom<HS>;
  using L = DkdvSmem<HS>;
  constexpr int ST = DKDV_STAGES, ST2 = DKDV_TSTAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_kv, bar_q_full[ST], bar_q_empty[ST], bar_qt_full[ST2], bar_qt_empty[ST2];
  __shared__ uint64_t bar_sdp[2], bar_pds[2], bar_acc[2], bar_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = p.T;
  const int kt = (int)(blockIdx.x / p.BH);          // causal: low key tiles have the longest walks
  const int bh = blockIdx.x % p.BH;
  const int b = bh / p.NH, h = bh % p.NH;
  const int k0 = kt * BQ;
  const int q_start = CAUSAL ? k0 : 0;
  const int n_q = (T - q_start + BS - 1) / BS;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&bar_q_full[s], 1);
      mbar_init(&bar_q_empty[s], 1 + NT);            // the S^T/dP^T MMAs and the transposer warps
    }
    for (int s = 0; s < ST2; ++s) {
      mbar_init(&bar_qt_full[s], NT);
      mbar_init(&bar_qt_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_sdp[i], 1);
      mbar_init(&bar_pds[i], 4);                // one arrival per warp
      mbar_init(&bar_acc[i], 1);
    }
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

  if (warp == 4) {
    // ------------------------------------------------------------ TMA loader
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar_kv, 2 * G::TILE_L);
      load_tile<HS, BQ>(smem + L::K_OFF, &map_kv, &bar_kv, p.C + h * HS, k0, b);
      load_tile<HS, BQ>(smem + L::V_OFF, &map_kv, &bar_kv, 2 * p.C + h * HS, k0, b);
      for (int i = 0; i < n_q; ++i) {
        const int st = i % ST;
        if (i >= ST && !mbar_wait(&bar_q_empty[st], ((i / ST) - 1) & 1, &abort_sh, gerr)) break;
        mbar_arrive_expect_tx(&bar_q_full[st], 2 * G::TILE_S);
        load_tile<HS, BS>(smem + L::Q_OFF + st * G::TILE_S, &map_qs, &bar_q_full[st], h * HS, q_start + i * BS, b);
        load_tile<HS, BS>(smem + L::DO_OFF + st * G::TILE_S, &map_dos, &bar_q_full[st], h * HS, q_start + i * BS,
                          b);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_st = make_idesc_tf32(BQ, BS, false, false);   // [128 keys] x [64 q]
      constexpr uint32_t idesc_acc = make_idesc_tf32(BQ, HS, false, false);  // B = [HS][64 q] K-major
      const uint64_t dK = make_sdesc(smem_u32(smem + L::K_OFF), 16, 1024, SWZ_128B);
      const uint64_t dV = make_sdesc(smem_u32(smem + L::V_OFF), 16, 1024, SWZ_128B);
      const uint64_t dQk = make_sdesc(smem_u32(smem + L::Q_OFF), 16, 1024, SWZ_128B);
      const uint64_t dOk = make_sdesc(smem_u32(smem + L::DO_OFF), 16, 1024, SWZ_128B);
      const uint64_t dQt = make_sdesc(smem_u32(smem + L::QT_OFF), 16, 1024, SWZ_128B);
      const uint64_t dOt = make_sdesc(smem_u32(smem + L::DOT_OFF), 16, 1024, SWZ_128B);
      // S^T(i) = K Q_i^T and dP^T(i) = V dO_i^T; releases the Q/dO stage when they finish
      auto issue_sdp = [&](int i) -> bool {
        if (!mbar_wait(&bar_q_full[i % ST], (i / ST) & 1, &abort_sh, gerr)) return false;
        tc_fence_after();
        const uint32_t so = (i % ST) * G::TILE_S, bb = (i & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < HS / 8; ++kk)
          mma_ss_tf32(tmem + bb, desc_add(dK, kmaj_step<G::BLK_L>(kk)), desc_add(dQk, so + kmaj_step<G::BLK_S>(kk)),
                      idesc_st, kk > 0);
#pragma unroll
        for (int kk = 0; kk < HS / 8; ++kk)
          mma_ss_tf32(tmem + 128 + bb, desc_add(dV, kmaj_step<G::BLK_L>(kk)),
                      desc_add(dOk, so + kmaj_step<G::BLK_S>(kk)), idesc_st, kk > 0);
        mma_commit(&bar_sdp[i & 1]);
        if (i + ST < n_q) mma_commit(&bar_q_empty[i % ST]);
        return true;
      };
      // dV += P^T(i) dO_i and dK += dS^T(i) Q_i (A from TMEM, B the transposed tiles)
      auto issue_acc = [&](int i) {
        const uint32_t so = (i % ST2) * G::TILE_S, bb = (i & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < BS / 8; ++kk)
          mma_ts_tf32(tmem + 256, tmem + bb + kk * 8, desc_add(dOt, so + kmaj_step<HS * 128>(kk)), idesc_acc,
                      (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BS / 8; ++kk)
          mma_ts_tf32(tmem + 320, tmem + 128 + bb + kk * 8, desc_add(dQt, so + kmaj_step<HS * 128>(kk)), idesc_acc,
                      (i > 0 || kk > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(&bar_kv, 0, &abort_sh, gerr);
      for (int ii = 0; ok && ii < 2 && ii < n_q; ++ii) ok = issue_sdp(ii);
      for (int i = 0; ok && i < n_q; ++i) {
        if (!(ok = mbar_wait(&bar_pds[i & 1], (i >> 1) & 1, &abort_sh, gerr))) break;
        if (!(ok = mbar_wait(&bar_qt_full[i % ST2], (i / ST2) & 1, &abort_sh, gerr))) break;
        tc_fence_after();
        issue_acc(i);
        if (i + ST2 < n_q) mma_commit(&bar_qt_empty[i % ST2]);
        if (i + 2 < n_q) {
          // the next scores of this buffer overwrite P^T(i), dS^T(i): wait for dV, dK
          // (committed only when awaited, so no arrival lands after the CTA retires)
          mma_commit(&bar_acc[i & 1]);
          if (!(ok = mbar_wait(&bar_acc[i & 1], (i >> 1) & 1, &abort_sh, gerr))) break;
          ok = issue_sdp(i + 2);
        }
      }
      if (ok) mma_commit(&bar_done);
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ Q / dO transposers
    const int wt = warp - 6;
    bool ok = true;
    for (int i = 0; ok && i < n_q; ++i) {
      const int st = i % ST, st2 = i % ST2;
      ok = mbar_wait(&bar_q_full[st], (i / ST) & 1, &abort_sh, gerr);
      if (ok && i >= ST2) ok = mbar_wait(&bar_qt_empty[st2], ((i / ST2) - 1) & 1, &abort_sh, gerr);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      for (int sb = wt; sb < 4 * G::NB; sb += NT) {
        const bool is_do = sb >= 2 * G::NB;
        const int x = is_do ? sb - 2 * G::NB : sb;
        transpose_sub<HS>(smem + (is_do ? L::DO_OFF : L::Q_OFF) + st * G::TILE_S,
                          smem + (is_do ? L::DOT_OFF : L::QT_OFF) + st2 * G::TILE_S, x, lane);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar_qt_full[st2]);
        if (i + ST < n_q) mbar_arrive(&bar_q_empty[st]);
      }
    }
  } else {
    // ------------------------------------------------------------ P^T / dS^T warpgroup (thread = key row)
    const int r = (warp << 5) + lane;
    const int kv = k0 + r;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float c = p.scale_log2;
    const float* lse_h = p.lse + (size_t)bh * T;
    const float* D_h = p.D + (size_t)bh * T;
    float* rows = reinterpret_cast<float*>(smem + L::ROW_OFF);
    bool ok = true;
    for (int i = 0; i < n_q; ++i) {
      const int bb = i & 1;
      const int q0 = q_start + i * BS;
      // this step's row statistics: threads 0-63 lse*log2e (+inf past T: P = 0), 64-127 D
      {
        const int q = q0 + (r & 63);
        float v;
        const bool in = q < T && ATTN_IN_RANGE((size_t)bh * T + q < (size_t)p.BH * T, gerr);
        if (r < 64) v = in ? __ldg(lse_h + q) * LOG2E : INFINITY;
        else v = in ? __ldg(D_h + q) : 0.f;
        rows[bb * 128 + r] = v;
      }
      // the barrier also shares a failure of any warp, so all leave together
      if (named_bar_red_or(1, 128, !ok)) { ok = false; break; }
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_sdp[bb], (i >> 1) & 1, &abort_sh, gerr));
      if (!ok) continue;
      tc_fence_after();
      uint32_t s[2][32], dp[2][32];
      tmem_ld64(tmem + lane_off + bb * 64, s);
      tmem_ld64(tmem + lane_off + 128 + bb * 64, dp);
      const float* rl = rows + bb * 128;
      const int lo = CAUSAL ? kv - q0 : -1;      // columns c < lo are masked (query before key)
      const float2 c2 = make_float2(c, c);
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(rl + q * 32 + e);
          const float4 d4 = *reinterpret_cast<const float4*>(rl + 64 + q * 32 + e);
          const float2 x0 = fma2(make_float2(__uint_as_float(s[q][e]), __uint_as_float(s[q][e + 1])), c2,
                                 make_float2(-l4.x, -l4.y));
          const float2 x1 = fma2(make_float2(__uint_as_float(s[q][e + 2]), __uint_as_float(s[q][e + 3])), c2,
                                 make_float2(-l4.z, -l4.w));
          float pv[4] = {ex2_approx(x0.x), ex2_approx(x0.y), ex2_approx(x1.x), ex2_approx(x1.y)};
          const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (CAUSAL && q * 32 + e + u < lo) pv[u] = 0.f;
            const float ds = pv[u] * (__uint_as_float(dp[q][e + u]) - dd[u]);
            s[q][e + u] = round_tf32(pv[u]);
            dp[q][e + u] = round_tf32(ds);
          }
        }
      tmem_st32(tmem + lane_off + bb * 64, s[0]);
      tmem_st32(tmem + lane_off + bb * 64 + 32, s[1]);
      tmem_st32(tmem + lane_off + 128 + bb * 64, dp[0]);
      tmem_st32(tmem + lane_off + 128 + bb * 64 + 32, dp[1]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pds[bb]);
    }
    ok = !named_bar_red_or(1, 128, !ok);
    if (ok) {
      // epilogue: dV and scale*dK through the (dead) V and K tiles, TMA-stored into dqkv
      const bool fail = !mbar_wait(&bar_done, 0, &abort_sh, gerr);
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < HS; cc += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + 256 + cc, v);
        tmem_ld_wait(v);
        stage32(smem + L::V_OFF, r, cc, v, 1.f);
        tmem_ld32(tmem + lane_off + 320 + cc, v);
        tmem_ld_wait(v);
        stage32(smem + L::K_OFF, r, cc, v, p.scale);
      }
      fence_proxy_async_smem();
      if (!named_bar_red_or(1, 128, fail) && warp == 0 && lane == 0) {
        store_tile<HS>(&map_g, smem + L::K_OFF, p.C + h * HS, k0, b);
        store_tile<HS>(&map_g, smem + L::V_OFF, 2 * p.C + h * HS, k0, b);
        bulk_commit_group();
        bulk_wait_group_read0();
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

// ============================================================================
// backward: dQ (one CTA per 128-row query tile)
// ============================================================================
// TMEM: S buffers [0,64) [64,128), dP buffers [128,192) [192,256) (dS in
// place), dQ [256, 256+HS).
// Warps: 0-3 dS (thread = query row), 4 TMA loader, 5 MMA issuer, 6-7 K transposers.
constexpr int DQ_STAGES = 3;      // K / V ring
constexpr int DQ_TSTAGES = 2;     // transposed K ring

template <int HS>
struct DqSmem {
  using G = Geom<HS>;
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = Q_OFF + G::TILE_L;
  static constexpr int K_OFF = DO_OFF + G::TILE_L;                 // DQ_STAGES tiles of 64 rows
  static constexpr int V_OFF = K_OFF + DQ_STAGES * G::TILE_S;
  static constexpr int KT_OFF = V_OFF + DQ_STAGES * G::TILE_S;     // DQ_TSTAGES [HS][64] tiles
  static constexpr int BYTES = KT_OFF + DQ_TSTAGES * G::TILE_S;
  static constexpr int ALLOC = BYTES + 1024;
};

template <int HS, bool CAUSAL>
__global__ void __launch_bounds__(BWD_THREADS, 1)
attn_bwd_dq_f32(const __grid_constant__ CUtensorMap map_ql, const __grid_constant__ CUtensorMap map_kvs,
                const __grid_constant__ CUtensorMap map_dol, const __grid_constant__ CUtensorMap map_g,
                const BwdParams p) {
  using G = Geom<HS>;
  using L = DqSmem<HS>;
  constexpr int ST = DQ_STAGES, ST2 = DQ_TSTAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_q, bar_kv_full[ST], bar_kv_empty[ST], bar_kt_full[ST2], bar_kt_empty[ST2];
  __shared__ uint64_t bar_sdp[2], bar_pds[2], bar_acc[2], bar_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = p.T;
  const int qt = p.n_tiles - 1 - (int)(blockIdx.x / p.BH);   // causal: late query tiles walk furthest
  const int bh = blockIdx.x % p.BH;
  const int b = bh / p.NH, h = bh % p.NH;
  const int q0 = qt * BQ;
  const int kend = CAUSAL ? min(q0 + BQ, T) : T;
  const int n_k = (kend + BS - 1) / BS;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&bar_q, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&bar_kv_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1 + NT);           // the S/dP MMAs and the transposer warps
    }
    for (int s = 0; s < ST2; ++s) {
      mbar_init(&bar_kt_full[s], NT);
      mbar_init(&bar_kt_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_sdp[i], 1);
      mbar_init(&bar_pds[i], 4);                // one arrival per warp
      mbar_init(&bar_acc[i], 1);
    }
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

  if (warp == 4) {
    // ------------------------------------------------------------ TMA loader
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar_q, 2 * G::TILE_L);
      load_tile<HS, BQ>(smem + L::Q_OFF, &map_ql, &bar_q, h * HS, q0, b);
      load_tile<HS, BQ>(smem + L::DO_OFF, &map_dol, &bar_q, h * HS, q0, b);
      for (int j = 0; j < n_k; ++j) {
        const int st = j % ST;
        if (j >= ST && !mbar_wait(&bar_kv_empty[st], ((j / ST) - 1) & 1, &abort_sh, gerr)) break;
        mbar_arrive_expect_tx(&bar_kv_full[st], 2 * G::TILE_S);
        load_tile<HS, BS>(smem + L::K_OFF + st * G::TILE_S, &map_kvs, &bar_kv_full[st], p.C + h * HS, j * BS, b);
        load_tile<HS, BS>(smem + L::V_OFF + st * G::TILE_S, &map_kvs, &bar_kv_full[st], 2 * p.C + h * HS, j * BS,
                          b);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc_tf32(BQ, BS, false, false);    // [128 q] x [64 keys]
      constexpr uint32_t idesc_dq = make_idesc_tf32(BQ, HS, false, false);   // B = K^T [HS][64 keys]
      const uint64_t dQ = make_sdesc(smem_u32(smem + L::Q_OFF), 16, 1024, SWZ_128B);
      const uint64_t dO = make_sdesc(smem_u32(smem + L::DO_OFF), 16, 1024, SWZ_128B);
      const uint64_t dKk = make_sdesc(smem_u32(smem + L::K_OFF), 16, 1024, SWZ_128B);
      const uint64_t dVk = make_sdesc(smem_u32(smem + L::V_OFF), 16, 1024, SWZ_128B);
      const uint64_t dKt = make_sdesc(smem_u32(smem + L::KT_OFF), 16, 1024, SWZ_128B);
      // S(j) = Q K_j^T and dP(j) = dO V_j^T; releases the K/V stage when they finish
      auto issue_sdp = [&](int j) -> bool {
        if (!mbar_wait(&bar_kv_full[j % ST], (j / ST) & 1, &abort_sh, gerr)) return false;
        tc_fence_after();
        const uint32_t so = (j % ST) * G::TILE_S, bb = (j & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < HS / 8; ++kk)
          mma_ss_tf32(tmem + bb, desc_add(dQ, kmaj_step<G::BLK_L>(kk)), desc_add(dKk, so + kmaj_step<G::BLK_S>(kk)),
                      idesc_s, kk > 0);
#pragma unroll
        for (int kk = 0; kk < HS / 8; ++kk)
          mma_ss_tf32(tmem + 128 + bb, desc_add(dO, kmaj_step<G::BLK_L>(kk)),
                      desc_add(dVk, so + kmaj_step<G::BLK_S>(kk)), idesc_s, kk > 0);
        mma_commit(&bar_sdp[j & 1]);
        if (j + ST < n_k) mma_commit(&bar_kv_empty[j % ST]);
        return true;
      };
      bool ok = mbar_wait(&bar_q, 0, &abort_sh, gerr);
      for (int jj = 0; ok && jj < 2 && jj < n_k; ++jj) ok = issue_sdp(jj);
      for (int j = 0; ok && j < n_k; ++j) {
        if (!(ok = mbar_wait(&bar_pds[j & 1], (j >> 1) & 1, &abort_sh, gerr))) break;
        if (!(ok = mbar_wait(&bar_kt_full[j % ST2], (j / ST2) & 1, &abort_sh, gerr))) break;
        tc_fence_after();
        // dQ += dS(j) K_j: A = dS from TMEM, B = K_j^T
        const uint32_t so = (j % ST2) * G::TILE_S, bb = (j & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < BS / 8; ++kk)
          mma_ts_tf32(tmem + 256, tmem + 128 + bb + kk * 8, desc_add(dKt, so + kmaj_step<HS * 128>(kk)), idesc_dq,
                      (j > 0 || kk > 0) ? 1u : 0u);
        if (j + ST2 < n_k) mma_commit(&bar_kt_empty[j % ST2]);
        if (j + 2 < n_k) {
          // dP(j+2) overwrites dS(j): wait until dQ += dS(j) K is done
          mma_commit(&bar_acc[j & 1]);
          if (!(ok = mbar_wait(&bar_acc[j & 1], (j >> 1) & 1, &abort_sh, gerr))) break;
          ok = issue_sdp(j + 2);
        }
      }
      if (ok) mma_commit(&bar_done);
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ K transposers
    const int wt = warp - 6;
    bool ok = true;
    for (int j = 0; ok && j < n_k; ++j) {
      const int st = j % ST, st2 = j % ST2;
      ok = mbar_wait(&bar_kv_full[st], (j / ST) & 1, &abort_sh, gerr);
      if (ok && j >= ST2) ok = mbar_wait(&bar_kt_empty[st2], ((j / ST2) - 1) & 1, &abort_sh, gerr);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      for (int sb = wt; sb < 2 * G::NB; sb += NT)
        transpose_sub<HS>(smem + L::K_OFF + st * G::TILE_S, smem + L::KT_OFF + st2 * G::TILE_S, sb, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar_kt_full[st2]);
        if (j + ST < n_k) mbar_arrive(&bar_kv_empty[st]);
      }
    }
  } else {
    // ------------------------------------------------------------ dS warpgroup (thread = query row)
    const int r = (warp << 5) + lane;
    const int t = q0 + r;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float c = p.scale_log2;
    const bool in = t < T && ATTN_IN_RANGE((size_t)bh * T + t < (size_t)p.BH * T, gerr);
    const float lse2 = in ? __ldg(p.lse + (size_t)bh * T + t) * LOG2E : 0.f;
    const float Dt = in ? __ldg(p.D + (size_t)bh * T + t) : 0.f;
    const float2 c2 = make_float2(c, c), nl2 = make_float2(-lse2, -lse2), nd2 = make_float2(-Dt, -Dt);
    bool ok = true;
    for (int j = 0; j < n_k; ++j) {
      const int bb = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_sdp[bb], (j >> 1) & 1, &abort_sh, gerr));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[2][32], dp[2][32];
      tmem_ld64(tmem + lane_off + bb * 64, s);
      tmem_ld64(tmem + lane_off + 128 + bb * 64, dp);
      const int kbase = j * BS;
      const int limit = CAUSAL ? min(t - kbase + 1, T - kbase) : T - kbase;   // keys [kbase, kbase+limit)
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 x = fma2(make_float2(__uint_as_float(s[q][e]), __uint_as_float(s[q][e + 1])), c2, nl2);
          float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          if (q * 32 + e >= limit) pv.x = 0.f;
          if (q * 32 + e + 1 >= limit) pv.y = 0.f;
          const float2 ds = mul2(pv, add2(make_float2(__uint_as_float(dp[q][e]), __uint_as_float(dp[q][e + 1])), nd2));
          dp[q][e] = round_tf32(ds.x);
          dp[q][e + 1] = round_tf32(ds.y);
        }
      tmem_st32(tmem + lane_off + 128 + bb * 64, dp[0]);
      tmem_st32(tmem + lane_off + 128 + bb * 64 + 32, dp[1]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pds[bb]);
    }
    ok = !named_bar_red_or(1, 128, !ok);
    if (ok) {
      // epilogue: scale * dQ through the (dead) Q tile, TMA-stored into dqkv[:, :, 0:C]
      const bool fail = !mbar_wait(&bar_done, 0, &abort_sh, gerr);
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < HS; cc += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + 256 + cc, v);
        tmem_ld_wait(v);
        stage32(smem + L::Q_OFF, r, cc, v, p.scale);
      }
      fence_proxy_async_smem();
      if (!named_bar_red_or(1, 128, fail) && warp == 0 && lane == 0) {
        store_tile<HS>(&map_g, smem + L::Q_OFF, h * HS, q0, b);
        bulk_commit_group();
        bulk_wait_group_read0();
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

// ============================================================================
// host launchers
// ============================================================================
template <class K>
static cudaError_t set_smem(K k, int bytes) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int HS, bool CAUSAL>
static cudaError_t fwd_t(const CUtensorMap& mq, const CUtensorMap& mkv, const CUtensorMap& mo,
                         const FwdParams& p, cudaStream_t s) {
  auto k = attn_fwd_f32_kernel<HS, CAUSAL>;
  cudaError_t e = set_smem(k, FwdSmem<HS>::ALLOC);
  if (e != cudaSuccess) return e;
  ProfileScope ps(K_FWD, s);
  k<<<p.BH * p.n_pairs, FWD_THREADS, FwdSmem<HS>::ALLOC, s>>>(mq, mkv, mo, p);
  return cudaGetLastError();
}

template <int HS, bool CAUSAL>
static cudaError_t bwd_t(const CUtensorMap& q_l, const CUtensorMap& q_s, const CUtensorMap& do_l,
                         const CUtensorMap& do_s, const CUtensorMap& g_l, const float* dout, const float* out,
                         float* ws_D, const BwdParams& p0, const Problem& pr, cudaStream_t s) {
  cudaError_t e;
  {
    ProfileScope ps(K_BWD_PRE, s);
    const long long n = (long long)pr.B * pr.T * pr.C / 4;
    attn_bwd_pre_f32<HS><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(dout, out, ws_D, pr.T, pr.C, pr.NH, n,
                                                                    device_error_word());
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  BwdParams p = p0;
  p.n_tiles = (pr.T + BQ - 1) / BQ;
  {
    auto k = attn_bwd_dkdv_f32<HS, CAUSAL>;
    if ((e = set_smem(k, DkdvSmem<HS>::ALLOC)) != cudaSuccess) return e;
    ProfileScope ps(K_BWD_MAIN, s);
    k<<<p.BH * p.n_tiles, BWD_THREADS, DkdvSmem<HS>::ALLOC, s>>>(q_l, q_s, do_s, g_l, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    auto k = attn_bwd_dq_f32<HS, CAUSAL>;
    if ((e = set_smem(k, DqSmem<HS>::ALLOC)) != cudaSuccess) return e;
    ProfileScope ps(K_BWD_DQ, s);
    k<<<p.BH * p.n_tiles, BWD_THREADS, DqSmem<HS>::ALLOC, s>>>(q_l, q_s, do_l, g_l, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace f32k

// map_q_l: qkv, box {32, 128}; map_q_s: qkv, box {32, 64}; map_out_l: out, box {32, 128}
cudaError_t launch_fwd_f32(const CUtensorMap& map_q_l, const CUtensorMap& map_q_s, const CUtensorMap& map_out_l,
                           float* lse, const Problem& pr, cudaStream_t stream) {
  f32k::FwdParams p;
  p.lse = lse;
  p.err = device_error_word();
  p.T = pr.T;
  p.NH = pr.NH;
  p.C = pr.C;
  p.BH = pr.B * pr.NH;
  p.n_pairs = (pr.T + 2 * f32k::BQ - 1) / (2 * f32k::BQ);
  p.scale_log2 = (1.0f / sqrtf((float)pr.hs)) * f32k::LOG2E;
  if (pr.hs == 64)
    return pr.causal ? f32k::fwd_t<64, true>(map_q_l, map_q_s, map_out_l, p, stream)
                     : f32k::fwd_t<64, false>(map_q_l, map_q_s, map_out_l, p, stream);
  return pr.causal ? f32k::fwd_t<32, true>(map_q_l, map_q_s, map_out_l, p, stream)
                   : f32k::fwd_t<32, false>(map_q_l, map_q_s, map_out_l, p, stream);
}

// map_q_l/_s: qkv boxes {32,128}/{32,64}; map_do_l/_s: dout; map_g_l: dqkv, box {32,128}
cudaError_t launch_bwd_f32(const CUtensorMap& map_q_l, const CUtensorMap& map_q_s, const CUtensorMap& map_do_l,
                           const CUtensorMap& map_do_s, const CUtensorMap& map_g_l, const float* dout,
                           const float* out, const float* lse, float* ws_D, const Problem& pr,
                           cudaStream_t stream) {
  f32k::BwdParams p;
  p.lse = lse;
  p.D = ws_D;
  p.err = device_error_word();
  p.T = pr.T;
  p.NH = pr.NH;
  p.C = pr.C;
  p.BH = pr.B * pr.NH;
  p.n_tiles = 0;
  p.scale = 1.0f / sqrtf((float)pr.hs);
  p.scale_log2 = p.scale * f32k::LOG2E;
  if (pr.hs == 64)
    return pr.causal
               ? f32k::bwd_t<64, true>(map_q_l, map_q_s, map_do_l, map_do_s, map_g_l, dout, out, ws_D, p, pr, stream)
               : f32k::bwd_t<64, false>(map_q_l, map_q_s, map_do_l, map_do_s, map_g_l, dout, out, ws_D, p, pr,
                                        stream);
  return pr.causal
             ? f32k::bwd_t<32, true>(map_q_l, map_q_s, map_do_l, map_do_s, map_g_l, dout, out, ws_D, p, pr, stream)
             : f32k::bwd_t<32, false>(map_q_l, map_q_s, map_do_l, map_do_s, map_g_l, dout, out, ws_D, p, pr, stream);
}

}  // namespace attn
