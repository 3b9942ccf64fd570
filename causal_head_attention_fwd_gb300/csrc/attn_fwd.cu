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
// Persistent: one CTA per SM. Work item = two 128-row query tiles of one
// (b, h) (256 rows); a CTA walks its items longest first (causal items are
// dealt by the host, each to the CTA with the least work so far; otherwise in
// a snake order over the CTAs). 12 warps:
//   warps 0-3  softmax warpgroup for query tile 0 (TMEM lanes 0-127)
//   warps 4-7  softmax warpgroup for query tile 1
//   warp  8    TMA producer: Q (double-buffered per item), K/V tiles through
//              a 4-stage ring that runs on across items
//   warps 9-10 MMA issuers, one thread per query tile; warp 11 idle
//   (setmaxnreg: 208 registers for the softmax warpgroups, 80 for warps 8-11)
// S_i(j+1) is issued as soon as the softmax warps of tile i hold S_i(j) in
// registers, so the next scores are ready when the softmax of this tile ends.
// The two softmax warpgroups take turns at the exponentials (two named
// barriers), so one forms P while the other loads its scores and takes its
// row maxima, instead of both sharing the MUFU at once.
// Each warpgroup writes its output tile through its own (then dead) Q tile and
// a TMA store while the next item's first scores are computed.
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+HS) O1 [320,320+HS)
//               P0 [384,448) P1 [448,512)  (P = bf16 pairs, 64 columns)
#include "common.cuh"
#include "fwd_deal.cuh"

namespace attn {

constexpr int FWD_STAGES = 4;
constexpr int FWD_THREADS = 384;
// register split: the two softmax warpgroups up, the producer/MMA warpgroup down
constexpr uint32_t FREG_SOFTMAX = 208, FREG_OTHER = 80;
static_assert(256 * FREG_SOFTMAX + 128 * FREG_OTHER <= 384 * 168, "register split exceeds the pool");
constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = 320, TM_P0 = 384, TM_P1 = 448;

template <int HS>
struct FwdSmem {
  static constexpr int TILE = TileGeom<HS>::TILE_BYTES;
  static constexpr int Q_OFF = 0;                          // 2 buffers x 2 tiles
  static constexpr int K_OFF = Q_OFF + 4 * TILE;           // FWD_STAGES tiles
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
  int n_items;         // n_pairs * BH
  float scale_log2;    // (1/sqrt(hs)) * log2(e)
};

struct FwdItem {
  int b, h, q0;
  int n_tile[2];       // key tiles each query tile sees (0: tile past T)
  int n_max;
};

template <bool CAUSAL>
__device__ __forceinline__ FwdItem fwd_decode(int idx, const FwdParams& p) {
  FwdItem w;
  const int pair = p.n_pairs - 1 - idx / p.BH;   // late (long causal rows) pairs first
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
__global__ void __launch_bounds__(FWD_THREADS, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap map_qkv,
                const __grid_constant__ CUtensorMap map_out, const FwdParams p,
                const __grid_constant__ WorkDeal sched) {
  using G = TileGeom<HS>;
  using L = FwdSmem<HS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_q_full[2], bar_q_empty[2];
  __shared__ uint64_t bar_k_full[FWD_STAGES], bar_v_full[FWD_STAGES], bar_kv_empty[FWD_STAGES];
  __shared__ uint64_t bar_s[2], bar_sfree[2], bar_p[2], bar_pv[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = p.T;
  // this CTA's items and its total number of key-tile steps
  const int n_items_cta = deal_count(sched, p.n_items);
  int total_kv = 0;
  for (int k = 0; k < n_items_cta; ++k) total_kv += fwd_decode<CAUSAL>(deal_item(sched, k), p).n_max;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_q_full[s], 1);
      mbar_init(&bar_q_empty[s], 2);             // one release per softmax warpgroup
    }
    for (int s = 0; s < FWD_STAGES; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_kv_empty[s], 2);            // one release per MMA issuer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s[i], 1);
      mbar_init(&bar_sfree[i], 4);               // one arrival per softmax warp
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
  pdl_launch_and_wait();

  if (warp >= 8) {
  setmaxnreg_dec<FREG_OTHER>();
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_qkv);
      bool ok = true;
      int gk = 0;                                 // key-tile steps so far
      FwdItem w_next = n_items_cta > 0 ? fwd_decode<CAUSAL>(deal_item(sched, 0), p) : FwdItem{};
      for (int ic = 0; ok && ic < n_items_cta; ++ic) {
        const FwdItem w = w_next;                 // decoded one item ahead
        if (ic + 1 < n_items_cta) w_next = fwd_decode<CAUSAL>(deal_item(sched, ic + 1), p);
        const int qb = ic & 1;
        if (ic >= 2 && !(ok = mbar_wait(&bar_q_empty[qb], ((ic >> 1) - 1) & 1, &abort_sh, gerr))) break;
        const uint32_t qbytes = (w.n_tile[0] > 0 ? G::TILE_BYTES : 0) + (w.n_tile[1] > 0 ? G::TILE_BYTES : 0);
        mbar_arrive_expect_tx(&bar_q_full[qb], qbytes);
        for (int i = 0; i < 2; ++i)
          if (w.n_tile[i] > 0)
            tma_load_3d(smem + L::Q_OFF + (2 * qb + i) * G::TILE_BYTES, &map_qkv, &bar_q_full[qb], w.h * HS,
                        w.q0 + i * BM, w.b);
        for (int j = 0; j < w.n_max; ++j, ++gk) {
          const int st = gk % FWD_STAGES;
          if (gk >= FWD_STAGES &&
              !(ok = mbar_wait(&bar_kv_empty[st], ((gk / FWD_STAGES) - 1) & 1, &abort_sh, gerr)))
            break;
          mbar_arrive_expect_tx(&bar_k_full[st], G::TILE_BYTES);
          tma_load_3d(smem + L::K_OFF + st * G::TILE_BYTES, &map_qkv, &bar_k_full[st], p.C + w.h * HS, j * BN, w.b);
          mbar_arrive_expect_tx(&bar_v_full[st], G::TILE_BYTES);
          tma_load_3d(smem + L::V_OFF + st * G::TILE_BYTES, &map_qkv, &bar_v_full[st], 2 * p.C + w.h * HS,
                      j * BN, w.b);
        }
      }
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers, one per query tile
    // Each tile has its own issuing thread, so S_i(j+1) is issued as soon as
    // softmax warpgroup i holds S_i(j), whatever the other tile is doing.
    if (lane == 0) {
      const int i = warp - 9;                     // query tile of this issuer
      constexpr uint32_t idesc_s = make_idesc_bf16(BM, BN, false, false);
      constexpr uint32_t idesc_o = make_idesc_bf16(BM, HS, false, true);
      const uint64_t dQ0 = make_sdesc(smem_u32(smem + L::Q_OFF), 16, G::ATOM_BYTES, G::SWZ);
      const uint64_t dK0 = make_sdesc(smem_u32(smem + L::K_OFF), 16, G::ATOM_BYTES, G::SWZ);
      const uint64_t dV0 = make_sdesc(smem_u32(smem + L::V_OFF), 16, G::ATOM_BYTES, G::SWZ);
      const uint32_t tS = tmem + (i ? TM_S1 : TM_S0), tO = tmem + (i ? TM_O1 : TM_O0), tP = tmem + (i ? TM_P1 : TM_P0);
      // S_i = Q_i K^T : K = HS in steps of 16 (32 bytes inside the swizzle row)
      auto issue_s = [&](int qb, int st) {
        const uint64_t qd = desc_add(dQ0, (2 * qb + i) * G::TILE_BYTES), kd = desc_add(dK0, st * G::TILE_BYTES);
#pragma unroll
        for (int k = 0; k < HS / 16; ++k) mma_ss(tS, desc_add(qd, k * 32), desc_add(kd, k * 32), idesc_s, k > 0);
        mma_commit(&bar_s[i]);
      };
      // O_i += P_i V : K = 128 keys in steps of 16 (16 rows of V = 2 atoms)
      auto issue_pv = [&](int st, bool acc) {
        const uint64_t vd = desc_add(dV0, st * G::TILE_BYTES);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ts(tO, tP + k * 8, desc_add(vd, k * 16 * G::ROW_BYTES), idesc_o, (acc || k > 0) ? 1u : 0u);
        mma_commit(&bar_pv[i]);
      };
      bool ok = true;
      int gk = 0;                                 // key-tile steps so far
      int gs = 0;                                 // softmax steps of this query tile so far
      FwdItem w_next = n_items_cta > 0 ? fwd_decode<CAUSAL>(deal_item(sched, 0), p) : FwdItem{};
      for (int ic = 0; ok && ic < n_items_cta; ++ic) {
        const FwdItem w = w_next;                 // decoded one item ahead
        if (ic + 1 < n_items_cta) w_next = fwd_decode<CAUSAL>(deal_item(sched, ic + 1), p);
        const int qb = ic & 1;
        const int n = w.n_tile[i];
        // first scores of the item, once the softmax warps hold the previous S_i
        if (n > 0) {
          if (!(ok = mbar_wait(&bar_q_full[qb], (ic >> 1) & 1, &abort_sh, gerr))) break;
          if (!(ok = mbar_wait(&bar_k_full[gk % FWD_STAGES], (gk / FWD_STAGES) & 1, &abort_sh, gerr))) break;
          if (gs > 0 && !(ok = mbar_wait(&bar_sfree[i], (gs - 1) & 1, &abort_sh, gerr))) break;
          tc_fence_after();
          issue_s(qb, gk % FWD_STAGES);
        }
        // per key tile j: S_i(j+1), then O_i += P_i(j) V_j
        for (int j = 0; ok && j < w.n_max; ++j) {
          const int st = (gk + j) % FWD_STAGES;
          const int st1 = (gk + j + 1) % FWD_STAGES;
          if (j + 1 < n) {
            if (!(ok = mbar_wait(&bar_sfree[i], (gs + j) & 1, &abort_sh, gerr))) break;
            if (!(ok = mbar_wait(&bar_k_full[st1], ((gk + j + 1) / FWD_STAGES) & 1, &abort_sh, gerr))) break;
            tc_fence_after();
            issue_s(qb, st1);
          }
          // every step, active or not, so this issuer never runs ahead of the
          // producer (the K/V stage release below needs both issuers)
          if (!(ok = mbar_wait(&bar_v_full[st], ((gk + j) / FWD_STAGES) & 1, &abort_sh, gerr))) break;
          if (j < n) {
            if (!(ok = mbar_wait(&bar_p[i], (gs + j) & 1, &abort_sh, gerr))) break;
            tc_fence_after();
            issue_pv(st, j > 0);
          }
          // release the K/V stage only if the producer will refill it (every
          // commit issued is awaited, so no arrival lands after the CTA retires)
          if (gk + j + FWD_STAGES < total_kv) mma_commit(&bar_kv_empty[st]);
        }
        gs += n;
        gk += w.n_max;
      }
    }
  }                                             // warp 11 only donates registers
  } else {
    setmaxnreg_inc<FREG_SOFTMAX>();
    // ------------------------------------------------------------ softmax warpgroups
    const int wg = warp >> 2;                    // query tile index 0/1
    const int r = ((warp & 3) << 5) + lane;      // row inside the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + (wg ? TM_S1 : TM_S0);
    const uint32_t tO = tmem + lane_off + (wg ? TM_O1 : TM_O0);
    const uint32_t tP = tmem + lane_off + (wg ? TM_P1 : TM_P0);
    const uint32_t bar_id = 1 + wg;              // named barrier of this warpgroup
    // The two warpgroups take turns at the exponentials (named barriers 3 and
    // 4, 256 threads), tile 1 first at every key step: one forms P while the
    // other waits for its scores and takes its row maxima, so the two tiles'
    // exponentials do not share the MUFU. Every warp takes one turn per key
    // step of every item (with no work where its tile has no such step or its
    // wait gave up), so the hand-overs always pair up. Tile 0's causal rows
    // end one key tile earlier; its spare turn follows tile 1's last step, so
    // tile 1 starts the next item without waiting for tile 0.
    const uint32_t my_turn = 3 + wg, next_turn = 4 - wg;
    auto idle_turns = [&](int k) {
      for (; k > 0; --k) {
        named_bar_sync(my_turn, 256);
        named_bar_arrive(next_turn, 256);
      }
    };
    const bool leader = (warp & 3) == 0 && lane == 0;
    const float c = p.scale_log2;
    bool ok = true;
    int gs = 0;                                  // softmax steps of this tile so far
    int q_pending = -1;                          // Q buffer still to hand back
    auto release_q = [&]() {
      if (q_pending >= 0 && leader) {
        bulk_wait_group_read0();
        mbar_arrive(&bar_q_empty[q_pending]);
      }
      q_pending = -1;
    };
    if (wg == 0) named_bar_arrive(4, 256);       // tile 1 takes the first turn
    FwdItem w_next = n_items_cta > 0 ? fwd_decode<CAUSAL>(deal_item(sched, 0), p) : FwdItem{};
    int ic = 0;
    for (; ok && ic < n_items_cta; ++ic) {
      const FwdItem w = w_next;                  // decoded one item ahead
      if (ic + 1 < n_items_cta) w_next = fwd_decode<CAUSAL>(deal_item(sched, ic + 1), p);
      const int qb = ic & 1;
      const int n = w.n_tile[wg];
      const int t = w.q0 + wg * BM + r;          // query row
      float m_run = -INFINITY, l_run = 0.f;
      int turns = 0;                             // turns taken in this item
      for (int j = 0; j < n; ++j) {
        const int gj = gs + j;
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
        if (lane == 0) mbar_arrive(&bar_sfree[wg]);      // S columns may be overwritten now
        // mask: causal diagonal tile (key > row), or keys past T (non-causal tail)
        const int kbase = j * BN;
        int limit = BN;                                  // keys [kbase, kbase+limit) are visible
        if (CAUSAL) { if (kbase + BN > t) limit = t - kbase + 1; }
        else { if (kbase + BN > T) limit = T - kbase; }
        if (__any_sync(0xffffffffu, limit < BN)) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (q * 32 + e >= limit) s[q][e] = __float_as_uint(-INFINITY);
        }
        // row max: 3-input max in 8 independent chains, then a short tree
        float mx8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            mx8[(e >> 1) & 7] = fmax3(mx8[(e >> 1) & 7], __uint_as_float(s[q][e]), __uint_as_float(s[q][e + 1]));
        const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        // Lazy rescaling: the exponent reference m_run only moves when the row
        // max exceeds it by more than 8 (log2 units), so p <= 2^8 and O is
        // rescaled rarely. Result and lse are exact for any reference value.
        const float m_new = (mx - m_run) * c > 8.f ? mx : m_run;
        const float alpha = ex2_approx((m_run - m_new) * c);
        const float2 c2 = make_float2(c, c), nmc = make_float2(-m_new * c, -m_new * c);
        float2 ls[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
        named_bar_sync(my_turn, 256);                    // this warpgroup's turn
        // p = exp2(s*c - m*c) in packed pairs; P goes to TMEM in two 64-key halves
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[32];
#pragma unroll
          for (int qq = 0; qq < 2; ++qq)
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int q = hf * 2 + qq;
              const float2 x = fma2(make_float2(__uint_as_float(s[q][e]), __uint_as_float(s[q][e + 1])), c2, nmc);
              const float2 ev = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              ls[(e >> 1) & 3] = add2(ls[(e >> 1) & 3], ev);
              pk[qq * 16 + e / 2] = pack_bf16x2(ev.x, ev.y);
            }
          if (hf == 0 && j > 0) {
            // P(j-1) must have been consumed (and O updated) by the previous P.V
            ok = __all_sync(0xffffffffu, mbar_wait(&bar_pv[wg], (gj - 1) & 1, &abort_sh, gerr));
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
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tmem_st32(tO + cc, o);
              }
            }
          }
          tmem_st32(tP + hf * 32, pk);
        }
        named_bar_arrive(next_turn, 256);                // the other warpgroup's turn
        ++turns;
        if (!ok) break;
        const float lsum = ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
        l_run = l_run * alpha + lsum;
        m_run = m_new;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p[wg]);
        if (j == 0) release_q();
      }
      idle_turns(w.n_max - turns);
      // -------------------------------------------------------- epilogue of this item
      // A warp whose wait gave up left the key loop early, but it still comes
      // here: failures are combined over the warpgroup at the barrier below, so
      // the four warps always leave together and none is left at a barrier.
      uint8_t* stage = smem + L::Q_OFF + (2 * qb + wg) * G::TILE_BYTES;   // this Q tile is dead now
      if (n > 0) {
        const bool fail = !ok || !mbar_wait(&bar_pv[wg], (gs + n - 1) & 1, &abort_sh, gerr);
        tc_fence_after();
        const float inv_l = 1.f / l_run;
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
        const size_t li = (size_t)(w.b * p.NH + w.h) * T + t;
        if (t < T && !fail && ATTN_IN_RANGE(li < (size_t)p.BH * T, gerr)) {
          // lse = scale*m + ln(l) = (m*c + log2 l) * ln 2
          p.lse[li] = (m_run * c + __log2f(l_run)) * 0.69314718055994531f;
        }
        fence_proxy_async_smem();
        if (named_bar_red_or(bar_id, 128, fail)) { ok = false; break; }
        if (leader) {
          tma_store_3d(&map_out, stage, w.h * HS, w.q0 + wg * BM, w.b);
          bulk_commit_group();
        }
      }
      release_q();
      if (ic + 2 < n_items_cta) q_pending = qb;
      gs += n;
    }
    // after a failure: the turns of the items not walked (the failed item's
    // were all taken before its epilogue)
    for (++ic; ic < n_items_cta; ++ic) idle_turns(fwd_decode<CAUSAL>(deal_item(sched, ic), p).n_max);
    if (wg == 1) named_bar_sync(4, 256);         // the other warpgroup's last hand-over
    if (leader) bulk_wait_group0();
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
                                const WorkDeal& sc, int grid, cudaStream_t stream) {
  auto k = attn_fwd_kernel<HS, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdSmem<HS>::ALLOC);
  if (e != cudaSuccess) return e;
  ProfileScope ps(K_FWD, stream);
  return launch_pdl(k, dim3(grid), dim3(FWD_THREADS), FwdSmem<HS>::ALLOC, stream, mq, mo, p, sc);
}

// The causal deal as plain arrays (see attn_fwd_schedule); 0 without a table.
int fwd_schedule(const Problem& pr, int n_cta, int* off, int* items, int cap) {
  const int n_pairs = (pr.T + 2 * BM - 1) / (2 * BM), BH = pr.B * pr.NH, n_items = n_pairs * BH;
  const int grid = n_items < n_cta ? n_items : n_cta;
  static thread_local WorkDeal s;
  build_causal_deal(s, n_pairs, BH, pr.T, grid);
  if (!s.use) return 0;
  if (cap < n_items) return -1;
  for (int c = 0; c <= grid; ++c) off[c] = s.off[c];
  for (int k = 0; k < n_items; ++k) items[k] = s.item[k];
  return n_items;
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
  p.n_items = p.n_pairs * p.BH;
  p.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)pr.hs));
  const int n_sm = device_sm_count();
  const int grid = p.n_items < n_sm ? p.n_items : n_sm;   // persistent: one CTA per SM
  const WorkDeal sc = launch_deal(pr.causal, p.n_pairs, p.BH, p.T, grid);
  if (pr.hs == 64)
    return pr.causal ? launch_fwd_t<64, true>(map_qkv, map_out, p, sc, grid, stream)
                     : launch_fwd_t<64, false>(map_qkv, map_out, p, sc, grid, stream);
  return pr.causal ? launch_fwd_t<32, true>(map_qkv, map_out, p, sc, grid, stream)
                   : launch_fwd_t<32, false>(map_qkv, map_out, p, sc, grid, stream);
}

}  // namespace attn
