// FP8 (e4m3) attention forward for sm_103a, on the GPT-2 (B, T, 3C) layout.
//
// The lower-precision forward that "LLM Systems 10 & 11: Accelerating
// Transformer Training and Inference", §1.3 (mixed-precision calculation)
// allows next to FP16: q, k, v are stored as e4m3 with one fp32 descale per
// 128-row tile of each head (real value = code * descale of its tile), the two
// contractions run on the tensor core as tcgen05.mma kind::f8f6f4 with fp32
// accumulation, and out is bf16. For query tile a and key tile b of a head,
// with dq_a, dk_b, dv_b the tiles' descales and dv* the largest dv_b the
// query tile sees:
//   y_tj  = scale log2(e) dq_a dk_b (q8_t . k8_j)     (exact fp32 sums of e4m3 products)
//   p'_tj = 2^(y_tj - m_t) (dv_b / dv*),  j in J(t)    (fp32, online; r_b = dv_b/dv* <= 1
//           folded into the exponent)
//   out_t = dv* sum_j e4m3(p'_tj) v8_j / sum_j p'_tj / r_b
//   lse_t = (m_t + log2 sum_j 2^(y_tj - m_t)) ln 2
// The probabilities enter P.V as e4m3 codes (p' <= 2^8 under the lazy
// rescaling below, inside e4m3's range of 448); the row sum uses the fp32 p.
//
// Same schedule as the bf16 forward (attention forward_cpu passes 1-4 of
// llm.c dev/cuda/attention_backward.cu, in the FlashAttention form of
// "Umakini wa kujitegemea, kerneli za CUDA na FlashAttention" section 3):
// persistent CTAs, work item = two 128-row query tiles of one (b, h), items
// dealt longest first as in fwd_deal.cuh, 12 warps
//   warps 0-3 / 4-7  softmax warpgroups of query tiles 0 / 1 (TMEM lanes);
//                    non-causal: taking turns at the exponentials
//   warp  8          TMA producer (Q per item, K/V through a ring)
//   warps 9-10       MMA issuers, one per query tile; warp 11 idle
// Tiles: [128 rows][hs] e4m3, hs bytes per row (64- or 32-byte swizzle). S and
// P.V use K = 32 per instruction; P lives in TMEM as 4 e4m3 codes per column.
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,320) O1 [320,384)
//               P0 [384,416) P1 [416,448)
#include "../../include/attn.h"
#include "common.cuh"
#include "fwd_deal.cuh"

namespace attn {
namespace f8 {

constexpr int STAGES = 4;
constexpr int THREADS = 384;
constexpr uint32_t REG_SOFTMAX = 208, REG_OTHER = 80;
static_assert(256 * REG_SOFTMAX + 128 * REG_OTHER <= 384 * 168, "register split exceeds the pool");
constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = 320, TM_P0 = 384, TM_P1 = 416;

// [128 rows][HS] e4m3 tile: HS bytes per row, swizzle atom 8 rows.
template <int HS>
struct Geom {
  static constexpr int ROW_BYTES = HS;
  static constexpr int ATOM_BYTES = 8 * HS;
  static constexpr uint32_t SWZ = HS == 64 ? SWZ_64B : SWZ_32B;
  static constexpr int TILE_BYTES = BM * HS;
};

template <int HS>
struct Smem {
  using G = Geom<HS>;
  static constexpr int OUT_TILE = BM * HS * 2;                  // bf16 [128][HS] staging
  static constexpr int Q_OFF = 0;                               // 2 buffers x 2 tiles
  static constexpr int K_OFF = Q_OFF + 4 * G::TILE_BYTES;       // STAGES tiles
  static constexpr int V_OFF = K_OFF + STAGES * G::TILE_BYTES;  // STAGES tiles
  static constexpr int OUT_OFF = V_OFF + STAGES * G::TILE_BYTES;   // 2 staging tiles
  static constexpr int BYTES = OUT_OFF + 2 * OUT_TILE;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
};

// Instruction descriptor, kind::f8f6f4 with e4m3 A and B (format code 0) and
// fp32 accumulation: bits 4-5 D format, 7-9 A format, 10-12 B format, bit 15/16
// A/B MN-major, 17-22 N>>3, 24-28 M>>4.
__host__ __device__ constexpr uint32_t make_idesc_e4m3(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_ss_e4m3(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_ts_e4m3(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// Four fp32 -> four e4m3 codes (round to nearest even, saturating), p0 in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float p0, float p1, float p2, float p3) {
  uint32_t w;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(w) : "f"(p0), "f"(p1), "f"(p2), "f"(p3));
  return w;
}

struct Params {
  float* lse;
  const float* descale;   // [3][B*NH][nT]: q, k, v descales per (head, 128-row tile)
  int* err;
  int T, NH, C;
  int nT;                 // 128-row tiles per head = ceil(T / 128)
  int n_pairs, BH, n_items;
  float scale_log2;       // (1/sqrt(hs)) * log2(e)
};

struct Item {
  int b, h, q0;
  int n_tile[2];
  int n_max;
};

template <bool CAUSAL>
__device__ __forceinline__ Item decode(int idx, const Params& p) {
  Item w;
  const int pair = p.n_pairs - 1 - idx / p.BH;   // long causal rows first
  const int bh = idx % p.BH;
  w.b = bh / p.NH;
  w.h = bh % p.NH;
  w.q0 = pair * 2 * BM;
  const int n_kv_all = (p.T + BN - 1) / BN;
  for (int i = 0; i < 2; ++i) {
    const int qs = w.q0 + i * BM;
    w.n_tile[i] = qs >= p.T ? 0 : (CAUSAL ? (qs / BN + 1) : n_kv_all);
  }
  w.n_max = w.n_tile[0] > w.n_tile[1] ? w.n_tile[0] : w.n_tile[1];
  return w;
}

template <int HS, bool CAUSAL>
__global__ void __launch_bounds__(THREADS, 1)
attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap map_qkv, const __grid_constant__ CUtensorMap map_out,
                    const Params p, const __grid_constant__ WorkDeal deal) {
  using G = Geom<HS>;
  using L = Smem<HS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_q_full[2], bar_q_empty[2];
  __shared__ uint64_t bar_k_full[STAGES], bar_v_full[STAGES], bar_kv_empty[STAGES];
  __shared__ uint64_t bar_s[2], bar_sfree[2], bar_p[2], bar_pv[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = p.T;
  // this CTA's items (longest first) and its total number of key-tile steps
  const int n_items_cta = deal_count(deal, p.n_items);
  int total_kv = 0;
  for (int k = 0; k < n_items_cta; ++k) total_kv += decode<CAUSAL>(deal_item(deal, k), p).n_max;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_q_full[s], 1);
      mbar_init(&bar_q_empty[s], 2);             // one release per softmax warpgroup
    }
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_kv_empty[s], 2);            // one release per MMA issuer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s[i], 1);
      mbar_init(&bar_sfree[i], 4);
      mbar_init(&bar_p[i], 4);
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

  if (warp >= 8) {
    setmaxnreg_dec<REG_OTHER>();
    if (warp == 8) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&map_qkv);
        bool ok = true;
        int gk = 0;
        for (int ic = 0; ok && ic < n_items_cta; ++ic) {
          const Item w = decode<CAUSAL>(deal_item(deal, ic), p);
          const int qb = ic & 1;
          if (ic >= 2 && !(ok = mbar_wait(&bar_q_empty[qb], ((ic >> 1) - 1) & 1, &abort_sh, gerr))) break;
          const uint32_t qbytes = (w.n_tile[0] > 0 ? G::TILE_BYTES : 0) + (w.n_tile[1] > 0 ? G::TILE_BYTES : 0);
          mbar_arrive_expect_tx(&bar_q_full[qb], qbytes);
          for (int i = 0; i < 2; ++i)
            if (w.n_tile[i] > 0)
              tma_load_3d(smem + L::Q_OFF + (2 * qb + i) * G::TILE_BYTES, &map_qkv, &bar_q_full[qb], w.h * HS,
                          w.q0 + i * BM, w.b);
          for (int j = 0; j < w.n_max; ++j, ++gk) {
            const int st = gk % STAGES;
            if (gk >= STAGES && !(ok = mbar_wait(&bar_kv_empty[st], ((gk / STAGES) - 1) & 1, &abort_sh, gerr)))
              break;
            mbar_arrive_expect_tx(&bar_k_full[st], G::TILE_BYTES);
            tma_load_3d(smem + L::K_OFF + st * G::TILE_BYTES, &map_qkv, &bar_k_full[st], p.C + w.h * HS, j * BN,
                        w.b);
            mbar_arrive_expect_tx(&bar_v_full[st], G::TILE_BYTES);
            tma_load_3d(smem + L::V_OFF + st * G::TILE_BYTES, &map_qkv, &bar_v_full[st], 2 * p.C + w.h * HS,
                        j * BN, w.b);
          }
        }
      }
    } else if (warp == 9 || warp == 10) {
      // ---------------------------------------------------------- MMA issuers
      if (lane == 0) {
        const int i = warp - 9;
        constexpr uint32_t idesc_s = make_idesc_e4m3(BM, BN, false, false);   // Q, K K-major
        constexpr uint32_t idesc_o = make_idesc_e4m3(BM, HS, false, true);    // P in TMEM, V MN-major
        const uint64_t dQ0 = make_sdesc(smem_u32(smem + L::Q_OFF), 16, G::ATOM_BYTES, G::SWZ);
        const uint64_t dK0 = make_sdesc(smem_u32(smem + L::K_OFF), 16, G::ATOM_BYTES, G::SWZ);
        const uint64_t dV0 = make_sdesc(smem_u32(smem + L::V_OFF), 16, G::ATOM_BYTES, G::SWZ);
        const uint32_t tS = tmem + (i ? TM_S1 : TM_S0), tO = tmem + (i ? TM_O1 : TM_O0), tP = tmem + (i ? TM_P1 : TM_P0);
        // S_i = Q_i K^T : K = HS in steps of 32 e4m3 (32 bytes inside the swizzle row)
        auto issue_s = [&](int qb, int st) {
          const uint64_t qd = desc_add(dQ0, (2 * qb + i) * G::TILE_BYTES), kd = desc_add(dK0, st * G::TILE_BYTES);
#pragma unroll
          for (int k = 0; k < HS / 32; ++k) mma_ss_e4m3(tS, desc_add(qd, k * 32), desc_add(kd, k * 32), idesc_s, k > 0);
          mma_commit(&bar_s[i]);
        };
        // O_i += P_i V : K = 128 keys in steps of 32 (32 rows of V, 8 TMEM columns of P)
        auto issue_pv = [&](int st, bool acc) {
          const uint64_t vd = desc_add(dV0, st * G::TILE_BYTES);
#pragma unroll
          for (int k = 0; k < BN / 32; ++k)
            mma_ts_e4m3(tO, tP + k * 8, desc_add(vd, k * 32 * G::ROW_BYTES), idesc_o, (acc || k > 0) ? 1u : 0u);
          mma_commit(&bar_pv[i]);
        };
        bool ok = true;
        int gk = 0, gs = 0;
        for (int ic = 0; ok && ic < n_items_cta; ++ic) {
          const Item w = decode<CAUSAL>(deal_item(deal, ic), p);
          const int qb = ic & 1;
          const int n = w.n_tile[i];
          if (n > 0) {
            if (!(ok = mbar_wait(&bar_q_full[qb], (ic >> 1) & 1, &abort_sh, gerr))) break;
            if (!(ok = mbar_wait(&bar_k_full[gk % STAGES], (gk / STAGES) & 1, &abort_sh, gerr))) break;
            if (gs > 0 && !(ok = mbar_wait(&bar_sfree[i], (gs - 1) & 1, &abort_sh, gerr))) break;
            tc_fence_after();
            issue_s(qb, gk % STAGES);
          }
          for (int j = 0; ok && j < w.n_max; ++j) {
            const int st = (gk + j) % STAGES;
            const int st1 = (gk + j + 1) % STAGES;
            if (j + 1 < n) {
              if (!(ok = mbar_wait(&bar_sfree[i], (gs + j) & 1, &abort_sh, gerr))) break;
              if (!(ok = mbar_wait(&bar_k_full[st1], ((gk + j + 1) / STAGES) & 1, &abort_sh, gerr))) break;
              tc_fence_after();
              issue_s(qb, st1);
            }
            // every step, active or not, so this issuer never runs ahead of the producer
            if (!(ok = mbar_wait(&bar_v_full[st], ((gk + j) / STAGES) & 1, &abort_sh, gerr))) break;
            if (j < n) {
              if (!(ok = mbar_wait(&bar_p[i], (gs + j) & 1, &abort_sh, gerr))) break;
              tc_fence_after();
              issue_pv(st, j > 0);
            }
            if (gk + j + STAGES < total_kv) mma_commit(&bar_kv_empty[st]);
          }
          gs += n;
          gk += w.n_max;
        }
      }
    }
  } else {
    setmaxnreg_inc<REG_SOFTMAX>();
    // ------------------------------------------------------------ softmax warpgroups
    const int wg = warp >> 2;
    const int r = ((warp & 3) << 5) + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + (wg ? TM_S1 : TM_S0);
    const uint32_t tO = tmem + lane_off + (wg ? TM_O1 : TM_O0);
    const uint32_t tP = tmem + lane_off + (wg ? TM_P1 : TM_P0);
    const uint32_t bar_id = 1 + wg;
    // Non-causal: turns at the exponentials, as in the bf16 forward (named
    // barriers 3 and 4, 256 threads, tile 1 first at every key step; every warp
    // takes one turn per key step of every item, with no work where it has
    // none). Causal items of 2-8 steps lost 2 us with them at the GPT-2 shape.
    constexpr bool TURNS = !CAUSAL;
    const uint32_t my_turn = 3 + wg, next_turn = 4 - wg;
    auto idle_turns = [&](int k) {
      if constexpr (TURNS) {
        for (; k > 0; --k) {
          named_bar_sync(my_turn, 256);
          named_bar_arrive(next_turn, 256);
        }
      }
    };
    const bool leader = (warp & 3) == 0 && lane == 0;
    uint8_t* stage = smem + L::OUT_OFF + wg * L::OUT_TILE;
    const size_t dstride = (size_t)p.BH * p.nT;  // between the q, k and v descale planes
    bool ok = true;
    int gs = 0;
    if (TURNS && wg == 0) named_bar_arrive(4, 256);   // tile 1 takes the first turn
    int ic = 0;
    for (; ok && ic < n_items_cta; ++ic) {
      const Item w = decode<CAUSAL>(deal_item(deal, ic), p);
      const int qb = ic & 1;
      const int n = w.n_tile[wg];
      const int t = w.q0 + wg * BM + r;
      // descales of this head: q of this query tile; k and v per key tile (the
      // head and its tiles lie inside the (3, B*NH, nT) array)
      const float* dsc = p.descale + (size_t)(w.b * p.NH + w.h) * p.nT;
      const bool dsc_in =
          ATTN_IN_RANGE(w.b * p.NH + w.h < p.BH && (n == 0 || (w.q0 + wg * BM) / BM < p.nT) && n <= p.nT, gerr);
      const float cq = n > 0 && dsc_in ? p.scale_log2 * __ldg(dsc + (w.q0 + wg * BM) / BM) : 0.f;
      float dv_ref = 0.f;                        // the largest v descale the tile sees
      for (int kt = 0; kt < n && dsc_in; ++kt) dv_ref = fmaxf(dv_ref, __ldg(dsc + 2 * dstride + kt));
      const float lg_dv_ref = __log2f(dv_ref);
      float m_run = -INFINITY, l_run = 0.f;
      int turns = 0;                             // turns taken in this item
      for (int j = 0; j < n; ++j) {
        const int gj = gs + j;
        // this key tile: exponent scale of the raw e4m3 products, and
        // log2(dv_j / dv*) <= 0, which puts V's descale into P
        const float c = dsc_in ? cq * __ldg(dsc + dstride + j) : 0.f;
        const float dvj = dsc_in ? __ldg(dsc + 2 * dstride + j) : 1.f;
        const float a_j = __log2f(dvj) - lg_dv_ref;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_s[wg], gj & 1, &abort_sh, gerr));
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_sfree[wg]);
        const int kbase = j * BN;
        int limit = BN;
        if (CAUSAL) { if (kbase + BN > t) limit = t - kbase + 1; }
        else { if (kbase + BN > T) limit = T - kbase; }
        if (__any_sync(0xffffffffu, limit < BN)) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (q * 32 + e >= limit) s[q][e] = __float_as_uint(-INFINITY);
        }
        float mx8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            mx8[(e >> 1) & 7] = fmax3(mx8[(e >> 1) & 7], __uint_as_float(s[q][e]), __uint_as_float(s[q][e + 1]));
        const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        // lazy rescaling: the reference max (log2 units, as y = s * c) moves
        // only when the row max exceeds it by more than 8, so p' <= p <= 2^8 < 448
        // (e4m3 range)
        const float my = mx * c;
        const float m_new = my - m_run > 8.f ? my : m_run;
        const float alpha = ex2_approx(m_run - m_new);
        const float2 c2 = make_float2(c, c), nmc = make_float2(a_j - m_new, a_j - m_new);
        float2 ls[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
        if (TURNS) named_bar_sync(my_turn, 256);         // this warpgroup's turn
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[16];
#pragma unroll
          for (int qq = 0; qq < 2; ++qq)
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const int q = hf * 2 + qq;
              const float2 x0 = fma2(make_float2(__uint_as_float(s[q][e]), __uint_as_float(s[q][e + 1])), c2, nmc);
              const float2 x1 =
                  fma2(make_float2(__uint_as_float(s[q][e + 2]), __uint_as_float(s[q][e + 3])), c2, nmc);
              const float2 e0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
              const float2 e1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
              ls[(e >> 2) & 3] = add2(ls[(e >> 2) & 3], add2(e0, e1));
              pk[qq * 8 + e / 4] = pack_e4m3x4(e0.x, e0.y, e1.x, e1.y);
            }
          if (hf == 0 && j > 0) {
            // P(j-1) must have been consumed (and O updated) by the previous P.V
            ok = __all_sync(0xffffffffu, mbar_wait(&bar_pv[wg], (gj - 1) & 1, &abort_sh, gerr));
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
          tmem_st16(tP + hf * 16, pk);
        }
        if (TURNS) named_bar_arrive(next_turn, 256);     // the other warpgroup's turn
        ++turns;
        if (!ok) break;
        const float lsum = ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
        l_run = l_run * alpha + lsum * ex2_approx(-a_j);   // the sum of p = p' / r_j
        m_run = m_new;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p[wg]);
      }
      idle_turns(w.n_max - turns);
      // ---------------------------------------------------------- epilogue of this item
      // A warp whose wait gave up left the key loop early, but it still comes
      // here: failures are combined over the warpgroup at the barrier below, so
      // the four warps always leave together and none is left at a barrier.
      if (n > 0) {
        const bool fail = !ok || !mbar_wait(&bar_pv[wg], (gs + n - 1) & 1, &abort_sh, gerr);
        tc_fence_after();
        const float f = dv_ref / l_run;
        // the previous item's store of this staging tile must have read it
        if (leader) bulk_wait_group_read0();
        if (named_bar_red_or(bar_id, 128, fail)) { ok = false; break; }
#pragma unroll
        for (int cc = 0; cc < HS; cc += 32) {
          uint32_t o[32];
          tmem_ld32(tO + cc, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[ch * 8 + 0]) * f, __uint_as_float(o[ch * 8 + 1]) * f);
            v.y = pack_bf16x2(__uint_as_float(o[ch * 8 + 2]) * f, __uint_as_float(o[ch * 8 + 3]) * f);
            v.z = pack_bf16x2(__uint_as_float(o[ch * 8 + 4]) * f, __uint_as_float(o[ch * 8 + 5]) * f);
            v.w = pack_bf16x2(__uint_as_float(o[ch * 8 + 6]) * f, __uint_as_float(o[ch * 8 + 7]) * f);
            *reinterpret_cast<uint4*>(stage + swz_chunk_offset<HS>(r, cc / 8 + ch)) = v;
          }
        }
        if (t < T && ATTN_IN_RANGE((size_t)(w.b * p.NH + w.h) * T + t < (size_t)p.BH * T, gerr))
          p.lse[(size_t)(w.b * p.NH + w.h) * T + t] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
        fence_proxy_async_smem();
        named_bar_sync(bar_id, 128);
        if (leader) {
          tma_store_3d(&map_out, stage, w.h * HS, w.q0 + wg * BM, w.b);
          bulk_commit_group();
        }
      }
      // the Q buffer is free once this tile's scores are done (all its MMAs have completed)
      if (leader && ic + 2 < n_items_cta) mbar_arrive(&bar_q_empty[qb]);
      gs += n;
    }
    // after a failure: the turns of the items not walked (the failed item's
    // were all taken before its epilogue)
    if (TURNS)
      for (++ic; ic < n_items_cta; ++ic) idle_turns(decode<CAUSAL>(deal_item(deal, ic), p).n_max);
    if (TURNS && wg == 1) named_bar_sync(4, 256);   // the other warpgroup's last hand-over
    if (leader) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (abort_sh) {
    for (int i = 0; i < 1000; ++i) __nanosleep(1000);
  }
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int HS, bool CAUSAL>
static cudaError_t launch_t(const CUtensorMap& mq, const CUtensorMap& mo, const Params& p, const WorkDeal& deal,
                            int grid, cudaStream_t stream) {
  auto k = attn_fwd_fp8_kernel<HS, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<HS>::ALLOC);
  if (e != cudaSuccess) return e;
  ProfileScope ps(K_FWD, stream);
  k<<<grid, THREADS, Smem<HS>::ALLOC, stream>>>(mq, mo, p, deal);
  return cudaGetLastError();
}

}  // namespace f8

// map_qkv: e4m3 qkv as bytes {3C, T, B}, box {hs, 128}, 64/32-byte swizzle;
// map_out: bf16 out {C, T, B}, box {hs, 128}, 128/64-byte swizzle.
cudaError_t launch_fwd_fp8(const CUtensorMap& map_qkv, const CUtensorMap& map_out, const float* descale, float* lse,
                           const Problem& pr, cudaStream_t stream) {
  f8::Params p;
  p.lse = lse;
  p.descale = descale;
  p.nT = (pr.T + BM - 1) / BM;
  p.err = device_error_word();
  p.T = pr.T;
  p.NH = pr.NH;
  p.C = pr.C;
  p.n_pairs = (pr.T + 2 * BM - 1) / (2 * BM);
  p.BH = pr.B * pr.NH;
  p.n_items = p.n_pairs * p.BH;
  p.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)pr.hs));
  const int n_sm = device_sm_count();
  const int grid = p.n_items < n_sm ? p.n_items : n_sm;
  const WorkDeal deal = launch_deal(pr.causal, p.n_pairs, p.BH, p.T, grid);
  if (pr.hs == 64)
    return pr.causal ? f8::launch_t<64, true>(map_qkv, map_out, p, deal, grid, stream)
                     : f8::launch_t<64, false>(map_qkv, map_out, p, deal, grid, stream);
  return pr.causal ? f8::launch_t<32, true>(map_qkv, map_out, p, deal, grid, stream)
                   : f8::launch_t<32, false>(map_qkv, map_out, p, deal, grid, stream);
}

}  // namespace attn

namespace attn {
namespace f8 {

// e4m3 codes -> bf16 values code * descale of the code's (part, head, 128-row
// tile), 16 codes per thread: one 16-byte load, two 16-byte stores. The 16
// codes of a thread lie in one head's slot (hs is a multiple of 16).
__global__ void attn_fp8_dequant(const uint4* __restrict__ codes, const float* __restrict__ descale,
                                 uint4* __restrict__ out, int T, int C, int NH, int BH, long long n16, int* err) {
  pdl_launch_and_wait();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const long long e = i * 16;                              // element index in (B, T, 3C)
  const long long row = e / (3LL * C);                     // b * T + t
  const int col = (int)(e - row * 3LL * C);
  const int part = col / C, h = (col - part * C) / (C / NH);
  const int b = (int)(row / T), t = (int)(row - (long long)b * T);
  const int nT = (T + BM - 1) / BM;
  const size_t di = ((size_t)part * BH + (size_t)b * NH + h) * nT + t / BM;
  if (!ATTN_IN_RANGE(di < 3 * (size_t)BH * nT, err)) return;
  const float d = __ldg(descale + di);
  const uint4 v = codes[i];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      // two e4m3 codes -> f16x2 (exact: e4m3 values are f16 values) -> f32 -> * descale -> bf16x2
      const uint16_t pair = (uint16_t)(w[k] >> (16 * hlf));
      uint32_t h2;
      asm("{\n\t.reg .b16 c;\n\tmov.b16 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h2) : "h"(pair));
      float lo, hi;
      asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
          : "=f"(lo), "=f"(hi) : "r"(h2));
      o[2 * k + hlf] = pack_bf16x2(lo * d, hi * d);
    }
  }
  out[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
  out[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace f8

cudaError_t launch_fp8_dequant(const void* codes, const float* descale, void* out, int B, int T, int C, int NH,
                               cudaStream_t stream) {
  const long long n16 = (long long)B * T * 3 * C / 16;
  const int threads = 256;
  const long long blocks = (n16 + threads - 1) / threads;
  return launch_pdl(f8::attn_fp8_dequant, dim3((unsigned)blocks), dim3(threads), 0, stream,
                    static_cast<const uint4*>(codes), descale, static_cast<uint4*>(out), T, C, NH, B * NH, n16,
                    device_error_word());
}

}  // namespace attn
