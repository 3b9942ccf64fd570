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
//   2. attn_bwd_kernel: persistent, one CTA per SM. Work item = (128-key tile,
//      b, h); a CTA walks its items (causal items dealt longest first, each to
//      the CTA with the least work so far, as the forward's; otherwise in a
//      snake order over the CTAs) and, per item, the query tiles that see
//      those keys. S, dP, dV, dK, dQ on tcgen05; dQ tiles are added into
//      the accumulator with TMA bulk reductions; dK/dV stored by TMA.
//      K is double-buffered, V refilled once an item's last dP is done, and
//      the Q/dO ring runs on across items, so the next item's loads and the
//      last item's dK/dV stores overlap compute.
//   3. attn_bwd_dq_out: dq accumulator -> bf16 into dqkv[:, :, 0:C].
//
// Main kernel: 16 warps.
//   warps 0-3   P/dS warpgroup A: keys [0, 64) of the tile, thread = query row
//   warps 4-7   P/dS warpgroup B: keys [64, 128)
//   warps 8-11  dQ warpgroup: thread = query row; TMEM -> smem -> TMA reduce-add;
//               after each item the dK/dV epilogue (thread = key row)
//   warp  12    loader: K per item (double-buffered), Q and dO per query tile
//               (3-stage ring)
//   warp  13    MMA issuer
//   warp  14    loader of V (one buffer, refilled once the item's last dP is done)
//   warp  15    idle
// With the query row as the thread (the TMEM lane of S = Q K^T and dP = dO V^T),
// the row statistics lse_t and D_t are two registers per thread, read from
// global memory one step ahead: the P/dS phase reads no shared memory. P and dS
// go to shared memory as [key block][query][64 keys] tiles, the MN-major A
// operands of dV += P^T dO and dK += dS^T Q; dS also goes to TMEM as the A
// operand of dQ = dS K.
// The P/dS warpgroups copy S/dP of step g into registers and release them at
// once, so the tensor core computes S/dP of step g+1 while P/dS of step g are
// formed. MMA order: S(g), dP(g), dK(g-1), dQ(g-1), dV(g-1).
// TMEM columns: S [0,128) dP [128,256) dV [256,320) dK [320,384) dQ [384,448)
//               dS [448,512) (bf16 pairs)
#include "common.cuh"
#include "fwd_deal.cuh"

namespace attn {

constexpr int BWD_STAGES = 3;
constexpr int BWD_THREADS = 512;
constexpr uint32_t TB_S = 0, TB_DP = 128, TB_DV = 256, TB_DK = 320, TB_DQ = 384, TB_DS = 448;
// register split: 2 P/dS warpgroups up, the other 2 warpgroups down.
// pool = 512 threads x 128 registers = 65536 = 256 x 160 + 256 x 96.
constexpr uint32_t REG_SOFTMAX = 160, REG_OTHER = 96;
static_assert(256 * REG_SOFTMAX + 256 * REG_OTHER <= 512 * 128, "register split exceeds the pool");

template <int HS>
struct BwdSmem {
  static constexpr int TILE = TileGeom<HS>::TILE_BYTES;
  static constexpr int K_OFF = 0;                              // 2 buffers
  static constexpr int V_OFF = K_OFF + 2 * TILE;               // 1 buffer
  static constexpr int Q_OFF = V_OFF + TILE;                   // BWD_STAGES tiles
  static constexpr int DO_OFF = Q_OFF + BWD_STAGES * TILE;     // BWD_STAGES tiles
  static constexpr int P_OFF = DO_OFF + BWD_STAGES * TILE;     // P: [2 key blocks][128 q][64 keys] bf16, SW128
  static constexpr int PT_BYTES = 2 * 128 * 128;
  static constexpr int DS_OFF = P_OFF + PT_BYTES;              // dS, same layout
  static constexpr int DQ_OFF = DS_OFF + PT_BYTES;             // dQ fp32 [128 q][32] SW128 block; dK/dV staging
  static constexpr int DQ_BYTES = 128 * 128;
  static constexpr int BYTES = DQ_OFF + DQ_BYTES;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(TILE <= DQ_BYTES, "dK/dV staging must fit in the dQ staging area");
  static_assert(P_OFF % 1024 == 0, "P/dS tiles must start on a 128-byte-swizzle atom");
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
};

struct BwdParams {
  const float* lse;   // (B, NH, T)
  const float* D;     // (B, NH, T)
  int* err;
  int T, NH, C;
  int n_kv;           // key tiles per head
  int BH;
  int n_items;        // n_kv * BH work items
  float scale;        // 1/sqrt(hs)
  float scale_log2;   // scale * log2(e)
};

struct BwdItem {
  int kv, bh, b, h, i0, n_it;
};

template <bool CAUSAL>
__device__ __forceinline__ BwdItem bwd_decode(int idx, const BwdParams& p) {
  BwdItem it;
  it.kv = idx / p.BH;                       // key tile; tile 0 (most causal work) first
  it.bh = idx % p.BH;
  it.b = it.bh / p.NH;
  it.h = it.bh % p.NH;
  it.i0 = CAUSAL ? it.kv : 0;               // first query tile that sees these keys
  it.n_it = (p.T + BM - 1) / BM - it.i0;
  return it;
}

// ----------------------------------------------------------------------------
// 1. D = rowsum(dout * out) per head; zero the dq accumulator.
//    One thread per 8 consecutive channels (16 bytes of bf16).
// ----------------------------------------------------------------------------
template <int HS>
__global__ void attn_bwd_pre(const uint4* __restrict__ dout, const uint4* __restrict__ out,
                             float* __restrict__ D, float4* __restrict__ dq_acc, int T, int C, int NH,
                             long long n_vec, int* err) {
  pdl_launch_and_wait();
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
    // the accumulator has 2 * n_vec float4s: zero two of them, each store
    // coalesced across the warp
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    dq_acc[i] = z;
    dq_acc[i + n_vec] = z;
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
    const long long di = (b * NH + h) * T + t;
    if (ATTN_IN_RANGE(di < n_vec * 8 / C * NH, err)) D[di] = acc;   // D has B*T*NH entries
  }
}

// ----------------------------------------------------------------------------
// 3. dq accumulator (fp32, already scaled) -> bf16 into dqkv[:, :, 0:C].
// ----------------------------------------------------------------------------
__global__ void attn_bwd_dq_out(const float4* __restrict__ dq_acc, uint4* __restrict__ dqkv, int C,
                                long long n_vec, int* err) {
  pdl_launch_and_wait();
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
  const long long oi = (bt * 3 * C + c) / 8;
  if (ATTN_IN_RANGE(oi < 3 * n_vec, err)) dqkv[oi] = v;              // dqkv has 3 * n_vec 16-byte chunks
  // The accumulator is dead now: drop its 128-byte lines from L2 without
  // writing them back (four threads read one line; n_vec is a multiple of 4).
  __syncwarp(__activemask());
  if ((i & 3) == 0) l2_discard128(dq_acc + 2 * i);
}

// ----------------------------------------------------------------------------
// P and dS of one query row over 64 keys (packed fp32 pair math):
//   P = exp2(s*c - lse*log2 e),   dS = P * (dP - D)
// nl = -lse*log2(e) of the row (-inf for rows past T, so P = 0 there), Dq its
// D. With MASK, keys at or past `lim` (causal diagonal, keys past T) give 0.
// ----------------------------------------------------------------------------
template <bool MASK>
__device__ __forceinline__ void bwd_p_ds(const uint32_t (&sv)[2][32], const uint32_t (&dpv)[2][32], float nl,
                                         float Dq, float c, int lim, uint32_t (&pk)[32], uint32_t (&dk)[32]) {
  const float2 c2 = make_float2(c, c), nl2 = make_float2(nl, nl), d2 = make_float2(Dq, Dq);
#pragma unroll
  for (int cq = 0; cq < 2; ++cq) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 s2 = make_float2(__uint_as_float(sv[cq][i]), __uint_as_float(sv[cq][i + 1]));
      const float2 dp2 = make_float2(__uint_as_float(dpv[cq][i]), __uint_as_float(dpv[cq][i + 1]));
      const float2 x = fma2(s2, c2, nl2);
      float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
      if (MASK) {
        const int col = cq * 32 + i;             // key index in this 64-key half
        if (col >= lim) e.x = 0.f;
        if (col + 1 >= lim) e.y = 0.f;
      }
      const float2 ds = mul2(e, sub2(dp2, d2));
      pk[cq * 16 + i / 2] = pack_bf16x2(e.x, e.y);
      dk[cq * 16 + i / 2] = pack_bf16x2(ds.x, ds.y);
    }
  }
}

// ----------------------------------------------------------------------------
// 2. main kernel
// ----------------------------------------------------------------------------
template <int HS, bool CAUSAL>
__global__ void __launch_bounds__(BWD_THREADS, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap map_qkv, const __grid_constant__ CUtensorMap map_dout,
                const __grid_constant__ CUtensorMap map_dqkv, const __grid_constant__ CUtensorMap map_dqacc,
                const BwdParams p, const __grid_constant__ WorkDeal sched) {
  using G = TileGeom<HS>;
  using L = BwdSmem<HS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_k_full[2], bar_k_empty[2], bar_v_full, bar_v_empty;
  __shared__ uint64_t bar_q_full[BWD_STAGES], bar_q_empty[BWD_STAGES];
  __shared__ uint64_t bar_sdp_full, bar_sdp_free, bar_pds_full, bar_ds_free, bar_p_free, bar_dq_free, bar_done,
      bar_epi_free;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = p.T;
  // this CTA's items and total number of steps (query tiles over all items)
  const int n_items_cta = deal_count(sched, p.n_items);
  int total_g = 0;
  for (int k = 0; k < n_items_cta; ++k) total_g += bwd_decode<CAUSAL>(deal_item(sched, k), p).n_it;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_k_empty[s], 1);
    }
    mbar_init(&bar_v_full, 1);
    mbar_init(&bar_v_empty, 1);
    for (int s = 0; s < BWD_STAGES; ++s) {
      mbar_init(&bar_q_full[s], 1);
      mbar_init(&bar_q_empty[s], 1);
    }
    mbar_init(&bar_sdp_full, 1);
    mbar_init(&bar_sdp_free, 8);                 // one arrival per P/dS warp
    mbar_init(&bar_pds_full, 8);
    mbar_init(&bar_ds_free, 1);                  // dK and dQ of the step done: dQ ready, dS free
    mbar_init(&bar_p_free, 1);                   // dV of the step read P
    mbar_init(&bar_dq_free, 4);                  // one arrival per dQ warp
    mbar_init(&bar_done, 1);
    mbar_init(&bar_epi_free, 4);
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
    setmaxnreg_dec<REG_OTHER>();
    if (warp == 12) {
      // ------------------------------------------------------------ loader: K, Q, dO
      if (lane == 0) {
        tma_prefetch_desc(&map_qkv);
        tma_prefetch_desc(&map_dout);
        bool ok = true;
        int g = 0;
        for (int ic = 0; ok && ic < n_items_cta; ++ic) {
          const BwdItem w = bwd_decode<CAUSAL>(deal_item(sched, ic), p);
          const int kb = ic & 1;
          if (ic >= 2 && !(ok = mbar_wait(&bar_k_empty[kb], ((ic >> 1) - 1) & 1, &abort_sh, gerr))) break;
          mbar_arrive_expect_tx(&bar_k_full[kb], G::TILE_BYTES);
          tma_load_3d(smem + L::K_OFF + kb * G::TILE_BYTES, &map_qkv, &bar_k_full[kb], p.C + w.h * HS, w.kv * BN, w.b);
          for (int it = 0; it < w.n_it; ++it, ++g) {
            const int st = g % BWD_STAGES;
            const int qi = w.i0 + it;
            if (g >= BWD_STAGES &&
                !(ok = mbar_wait(&bar_q_empty[st], ((g / BWD_STAGES) - 1) & 1, &abort_sh, gerr)))
              break;
            mbar_arrive_expect_tx(&bar_q_full[st], 2 * G::TILE_BYTES);
            tma_load_3d(smem + L::Q_OFF + st * G::TILE_BYTES, &map_qkv, &bar_q_full[st], w.h * HS, qi * BM, w.b);
            tma_load_3d(smem + L::DO_OFF + st * G::TILE_BYTES, &map_dout, &bar_q_full[st], w.h * HS, qi * BM, w.b);
          }
        }
      }
    } else if (warp == 14) {
      // ------------------------------------------------------------ loader: V
      if (lane == 0) {
        for (int ic = 0; ic < n_items_cta; ++ic) {
          const BwdItem w = bwd_decode<CAUSAL>(deal_item(sched, ic), p);
          // the previous item's dP steps must be done with the buffer
          if (ic >= 1 && !mbar_wait(&bar_v_empty, (ic - 1) & 1, &abort_sh, gerr)) break;
          mbar_arrive_expect_tx(&bar_v_full, G::TILE_BYTES);
          tma_load_3d(smem + L::V_OFF, &map_qkv, &bar_v_full, 2 * p.C + w.h * HS, w.kv * BN, w.b);
        }
      }
    } else if (warp == 13) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t id_s = make_idesc_bf16(BM, BN, false, false);     // [q x keys], K = HS, both K-major
        constexpr uint32_t id_acc = make_idesc_bf16(BN, HS, true, true);     // [keys x HS], K = q: A, B MN-major
        constexpr uint32_t id_dq = make_idesc_bf16(BM, HS, false, true);     // [q x HS], K = keys: A TMEM, B MN-major
        const uint64_t dK0 = make_sdesc(smem_u32(smem + L::K_OFF), 16, G::ATOM_BYTES, G::SWZ);
        const uint64_t dV0 = make_sdesc(smem_u32(smem + L::V_OFF), 16, G::ATOM_BYTES, G::SWZ);
        const uint64_t dQ0 = make_sdesc(smem_u32(smem + L::Q_OFF), 16, G::ATOM_BYTES, G::SWZ);
        const uint64_t dO0 = make_sdesc(smem_u32(smem + L::DO_OFF), 16, G::ATOM_BYTES, G::SWZ);
        // P^T, dS^T as MN-major A operands: M = keys, two 64-key atoms LBO = 16 KB
        // apart, K = queries in rows of 128 bytes (SBO = 8 rows)
        const uint64_t dPm = make_sdesc(smem_u32(smem + L::P_OFF), 16384, 1024, SWZ_128B);
        const uint64_t dSm = make_sdesc(smem_u32(smem + L::DS_OFF), 16384, 1024, SWZ_128B);
        // the step whose dK/dQ/dV are still to be issued
        struct Pend { int g, st, kb, ic; bool first, last; };
        bool ok = true;
        auto finish = [&](const Pend& f) -> bool {
          const uint64_t qd = desc_add(dQ0, f.st * G::TILE_BYTES), od = desc_add(dO0, f.st * G::TILE_BYTES);
          if (!mbar_wait(&bar_pds_full, f.g & 1, &abort_sh, gerr)) return false;
          // dK/dV of the previous item must have been read out by its epilogue
          if (f.first && f.ic > 0 && !mbar_wait(&bar_epi_free, (f.ic - 1) & 1, &abort_sh, gerr)) return false;
          tc_fence_after();
          // dK += dS^T Q  (K = 128 queries: 16 rows of the dS tile per instruction)
#pragma unroll
          for (int k = 0; k < BM / 16; ++k)
            mma_ss(tmem + TB_DK, desc_add(dSm, k * 16 * 128), desc_add(qd, k * 16 * G::ROW_BYTES), id_acc,
                   (!f.first || k > 0) ? 1u : 0u);
          if (f.g > 0) {
            if (!mbar_wait(&bar_dq_free, (f.g - 1) & 1, &abort_sh, gerr)) return false;
            tc_fence_after();
          }
          // dQ = dS K  (A = dS from TMEM, K = 128 keys = 64 columns of bf16 pairs)
          const uint64_t kd = desc_add(dK0, f.kb * G::TILE_BYTES);
#pragma unroll
          for (int k = 0; k < BN / 16; ++k)
            mma_ts(tmem + TB_DQ, tmem + TB_DS + k * 8, desc_add(kd, k * 16 * G::ROW_BYTES), id_dq, k > 0);
          // dQ is ready and dS (smem and TMEM) free once dK and dQ are done: the
          // dQ warps drain dQ and the P/dS warps write the next dS while dV runs
          mma_commit(&bar_ds_free);
          // dV += P^T dO
#pragma unroll
          for (int k = 0; k < BM / 16; ++k)
            mma_ss(tmem + TB_DV, desc_add(dPm, k * 16 * 128), desc_add(od, k * 16 * G::ROW_BYTES), id_acc,
                   (!f.first || k > 0) ? 1u : 0u);
          if (f.g + 1 < total_g) mma_commit(&bar_p_free);
          if (f.g + BWD_STAGES < total_g) mma_commit(&bar_q_empty[f.st]);
          if (f.last) {
            mma_commit(&bar_done);                           // dK/dV of item f.ic final
            if (f.ic + 2 < n_items_cta) mma_commit(&bar_k_empty[f.kb]);
          }
          return true;
        };
        Pend pend{0, 0, 0, 0, false, false};
        bool have_pend = false;
        int g = 0;
        for (int ic = 0; ok && ic < n_items_cta; ++ic) {
          const BwdItem w = bwd_decode<CAUSAL>(deal_item(sched, ic), p);
          const int kb = ic & 1;
          if (!(ok = mbar_wait(&bar_k_full[kb], (ic >> 1) & 1, &abort_sh, gerr))) break;
          if (!(ok = mbar_wait(&bar_v_full, ic & 1, &abort_sh, gerr))) break;
          const uint64_t kd = desc_add(dK0, kb * G::TILE_BYTES);
          for (int it = 0; ok && it < w.n_it; ++it, ++g) {
            const int st = g % BWD_STAGES;
            if (!(ok = mbar_wait(&bar_q_full[st], (g / BWD_STAGES) & 1, &abort_sh, gerr))) break;
            if (g > 0 && !(ok = mbar_wait(&bar_sdp_free, (g - 1) & 1, &abort_sh, gerr))) break;
            tc_fence_after();
            const uint64_t qd = desc_add(dQ0, st * G::TILE_BYTES), od = desc_add(dO0, st * G::TILE_BYTES);
            // S = Q K^T ; dP = dO V^T   (K-dim = HS, both operands K-major)
#pragma unroll
            for (int k = 0; k < HS / 16; ++k)
              mma_ss(tmem + TB_S, desc_add(qd, k * 32), desc_add(kd, k * 32), id_s, k > 0);
#pragma unroll
            for (int k = 0; k < HS / 16; ++k)
              mma_ss(tmem + TB_DP, desc_add(od, k * 32), desc_add(dV0, k * 32), id_s, k > 0);
            mma_commit(&bar_sdp_full);
            // V is free for the next item once this item's last dP is done
            if (it == w.n_it - 1 && ic + 1 < n_items_cta) mma_commit(&bar_v_empty);
            if (have_pend) ok = finish(pend);
            pend = Pend{g, st, kb, ic, it == 0, it == w.n_it - 1};
            have_pend = true;
          }
        }
        if (ok && have_pend) ok = finish(pend);
      }
    } else if (warp < 12) {
      // ------------------------------------------------------------ dQ warpgroup
      const int wq = warp - 8;
      const int r = (wq << 5) + lane;                // query row (dQ) / key row (dK, dV)
      const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
      const bool leader = (wq == 0 && lane == 0);
      uint8_t* sdq = smem + L::DQ_OFF;
      const float s = p.scale;
      int g = 0;
      bool ok = true;
      for (int ic = 0; ok && ic < n_items_cta; ++ic) {
        const BwdItem w = bwd_decode<CAUSAL>(deal_item(sched, ic), p);
        for (int it = 0; it < w.n_it; ++it, ++g) {
          const int qi = w.i0 + it;
          // failures are combined over the warpgroup at the first barrier, so a
          // bounded wait that gave up never leaves a thread stuck at a barrier
          const bool fail = !mbar_wait(&bar_ds_free, g & 1, &abort_sh, gerr);
          tc_fence_after();
          // one 32-column block at a time: TMEM -> 16 KB staging tile -> reduce;
          // the dQ columns are released once the last block is in registers
#pragma unroll
          for (int cc = 0; cc < HS / 32; ++cc) {
            uint32_t a[32];
            tmem_ld32(tmem + lane_off + TB_DQ + cc * 32, a);
            tmem_ld_wait(a);
            if (cc == HS / 32 - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bar_dq_free);
            }
            // the previous bulk operation must have finished reading the staging tile
            if (leader) bulk_wait_group_read0();
            if (named_bar_red_or(1, 128, fail)) { ok = false; break; }
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {           // [128 q][32 fp32], 128-byte swizzle
              const float4 v = make_float4(__uint_as_float(a[ch * 4 + 0]) * s, __uint_as_float(a[ch * 4 + 1]) * s,
                                           __uint_as_float(a[ch * 4 + 2]) * s, __uint_as_float(a[ch * 4 + 3]) * s);
              *reinterpret_cast<float4*>(sdq + swz_chunk_offset<64>(r, ch)) = v;
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (leader) {
              tma_reduce_add_3d(&map_dqacc, sdq, w.h * HS + cc * 32, qi * BM, w.b);
              bulk_commit_group();
            }
          }
          if (!ok) break;
        }
        if (!ok) break;
        // ---------------------------------------------------------- dK, dV of this item
        // dV goes to the staging tile and scale*dK to registers (bf16 pairs)
        // before either is stored, so the TMEM columns are handed back to the
        // next item's first dK and dV without waiting for the stores.
        const bool fail = !mbar_wait(&bar_done, ic & 1, &abort_sh, gerr);
        tc_fence_after();
        if (leader) bulk_wait_group_read0();             // staging free
        if (named_bar_red_or(1, 128, fail)) { ok = false; break; }
        uint8_t* stage = sdq;
#pragma unroll
        for (int cc = 0; cc < HS; cc += 16) {
          uint32_t o[16];
          tmem_ld16_wait(tmem + lane_off + TB_DV + cc, o);
          uint4 v0, v1;
          v0.x = pack_bf16x2(__uint_as_float(o[0]), __uint_as_float(o[1]));
          v0.y = pack_bf16x2(__uint_as_float(o[2]), __uint_as_float(o[3]));
          v0.z = pack_bf16x2(__uint_as_float(o[4]), __uint_as_float(o[5]));
          v0.w = pack_bf16x2(__uint_as_float(o[6]), __uint_as_float(o[7]));
          v1.x = pack_bf16x2(__uint_as_float(o[8]), __uint_as_float(o[9]));
          v1.y = pack_bf16x2(__uint_as_float(o[10]), __uint_as_float(o[11]));
          v1.z = pack_bf16x2(__uint_as_float(o[12]), __uint_as_float(o[13]));
          v1.w = pack_bf16x2(__uint_as_float(o[14]), __uint_as_float(o[15]));
          *reinterpret_cast<uint4*>(stage + swz_chunk_offset<HS>(r, cc / 8)) = v0;
          *reinterpret_cast<uint4*>(stage + swz_chunk_offset<HS>(r, cc / 8 + 1)) = v1;
        }
        uint32_t dkp[HS / 2];
#pragma unroll
        for (int cc = 0; cc < HS; cc += 16) {
          uint32_t o[16];
          tmem_ld16_wait(tmem + lane_off + TB_DK + cc, o);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dkp[cc / 2 + e] = pack_bf16x2(__uint_as_float(o[2 * e]) * s, __uint_as_float(o[2 * e + 1]) * s);
        }
        tc_fence_before();
        // every commit is awaited: only signal if the MMA warp will wait for it
        __syncwarp();
        if (lane == 0 && ic + 1 < n_items_cta) mbar_arrive(&bar_epi_free);   // dK/dV TMEM columns free
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          tma_store_3d(&map_dqkv, stage, 2 * p.C + w.h * HS, w.kv * BN, w.b);
          bulk_commit_group();
          bulk_wait_group_read0();                       // staging free again
        }
        named_bar_sync(1, 128);
#pragma unroll
        for (int ch = 0; ch < HS / 8; ++ch)
          *reinterpret_cast<uint4*>(stage + swz_chunk_offset<HS>(r, ch)) =
              make_uint4(dkp[ch * 4 + 0], dkp[ch * 4 + 1], dkp[ch * 4 + 2], dkp[ch * 4 + 3]);
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          tma_store_3d(&map_dqkv, stage, p.C + w.h * HS, w.kv * BN, w.b);
          bulk_commit_group();
        }
      }
      if (leader) bulk_wait_group0();
    }
  } else {
    setmaxnreg_inc<REG_SOFTMAX>();
    // ------------------------------------------------------------ P/dS warpgroups
    const int half = warp >> 2;                    // keys [64*half, 64*half+64) of the tile
    const int r = ((warp & 3) << 5) + lane;        // query row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float c = p.scale_log2;
    const float nlog2e = -1.4426950408889634f;
    uint8_t* sp = smem + L::P_OFF + half * 16384;
    uint8_t* sds = smem + L::DS_OFF + half * 16384;
    // this row's -lse*log2(e) and D for a (head, query tile): rows past T give P = 0
    auto load_row = [&](int bh, int qi, float& nl, float& dd) {
      const int q = qi * BM + r;
      const size_t i = (size_t)bh * T + q;
      const bool in = q < T && ATTN_IN_RANGE(i < (size_t)p.BH * T, gerr);
      nl = in ? __ldg(p.lse + i) * nlog2e : -INFINITY;
      dd = in ? __ldg(p.D + i) : 0.f;
    };
    float nl_next = 0.f, d_next = 0.f;
    if (n_items_cta > 0) {
      const BwdItem f = bwd_decode<CAUSAL>(deal_item(sched, 0), p);
      load_row(f.bh, f.i0, nl_next, d_next);
    }
    int g = 0;
    bool ok = true;
    for (int ic = 0; ok && ic < n_items_cta; ++ic) {
      const BwdItem w = bwd_decode<CAUSAL>(deal_item(sched, ic), p);
      for (int it = 0; it < w.n_it; ++it, ++g) {
        const int qi = w.i0 + it;
        const float nl = nl_next, dq = d_next;
        // the row statistics of the next step, loaded one step ahead
        if (it + 1 < w.n_it) {
          load_row(w.bh, qi + 1, nl_next, d_next);
        } else if (ic + 1 < n_items_cta) {
          const BwdItem nx = bwd_decode<CAUSAL>(deal_item(sched, ic + 1), p);
          load_row(nx.bh, nx.i0, nl_next, d_next);
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_sdp_full, g & 1, &abort_sh, gerr));
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[2][32], dpv[2][32];
        tmem_ld32(tmem + lane_off + TB_S + half * 64, sv[0]);
        tmem_ld32(tmem + lane_off + TB_S + half * 64 + 32, sv[1]);
        tmem_ld32(tmem + lane_off + TB_DP + half * 64, dpv[0]);
        tmem_ld32(tmem + lane_off + TB_DP + half * 64 + 32, dpv[1]);
        tmem_ld_wait(sv[0]);
        tmem_tie32(sv[1]);
        tmem_tie32(dpv[0]);
        tmem_tie32(dpv[1]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_sdp_free);   // S/dP columns may be overwritten now
        // keys [kbase, kbase + lim) of this half are visible to the row
        const int kbase = w.kv * BN + half * 64;
        int lim = 64;
        if (CAUSAL && qi == w.kv) lim = min(lim, r - half * 64 + 1);     // diagonal tile: key <= query
        if (kbase + 64 > T) lim = min(lim, T - kbase);                   // keys past T
        uint32_t pk[32], dk[32];
        if (__any_sync(0xffffffffu, lim < 64))
          bwd_p_ds<true>(sv, dpv, nl, dq, c, lim, pk, dk);
        else
          bwd_p_ds<false>(sv, dpv, nl, dq, c, 64, pk, dk);
        // dS into TMEM (A of dQ) and smem (A of dK), once the previous step's
        // dK and dQ have read them
        if (g > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_ds_free, (g - 1) & 1, &abort_sh, gerr));
          if (!ok) break;
          tc_fence_after();
        }
        tmem_st32(tmem + lane_off + TB_DS + half * 32, dk);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 v = make_uint4(dk[ch * 4 + 0], dk[ch * 4 + 1], dk[ch * 4 + 2], dk[ch * 4 + 3]);
          *reinterpret_cast<uint4*>(sds + swz_chunk_offset<64>(r, ch)) = v;
        }
        // P into smem (A of dV) once the previous step's dV has read it
        if (g > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_p_free, (g - 1) & 1, &abort_sh, gerr));
          if (!ok) break;
        }
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 v = make_uint4(pk[ch * 4 + 0], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
          *reinterpret_cast<uint4*>(sp + swz_chunk_offset<64>(r, ch)) = v;
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_pds_full);
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
                                   const CUtensorMap& macc, const BwdParams& p, const WorkDeal& deal, int grid,
                                   cudaStream_t stream) {
  auto k = attn_bwd_kernel<HS, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdSmem<HS>::ALLOC);
  if (e != cudaSuccess) return e;
  ProfileScope ps(K_BWD_MAIN, stream);
  return launch_pdl(k, dim3(grid), dim3(BWD_THREADS), BwdSmem<HS>::ALLOC, stream, mq, md, mg, macc, p, deal);
}

cudaError_t launch_bwd_bf16(const CUtensorMap& map_qkv, const CUtensorMap& map_dout,
                            const CUtensorMap& map_dqkv, const CUtensorMap& map_dqacc, const void* dout,
                            const void* out, const float* lse, void* dqkv, float* ws_D, float* ws_dq,
                            const Problem& pr, cudaStream_t stream) {
  const long long n_vec = (long long)pr.B * pr.T * pr.C / 8;
  const int threads = 256;
  const long long blocks = (n_vec + threads - 1) / threads;
  cudaError_t e;
  {
    ProfileScope ps(K_BWD_PRE, stream);
    e = launch_pdl(pr.hs == 64 ? attn_bwd_pre<64> : attn_bwd_pre<32>, dim3((unsigned)blocks), dim3(threads), 0,
                   stream, static_cast<const uint4*>(dout), static_cast<const uint4*>(out), ws_D,
                   reinterpret_cast<float4*>(ws_dq), pr.T, pr.C, pr.NH, n_vec, device_error_word());
  }
  if (e != cudaSuccess) return e;

  BwdParams p;
  p.lse = lse;
  p.D = ws_D;
  p.err = device_error_word();
  p.T = pr.T;
  p.NH = pr.NH;
  p.C = pr.C;
  p.n_kv = (pr.T + BN - 1) / BN;
  p.BH = pr.B * pr.NH;
  p.n_items = p.n_kv * p.BH;
  p.scale = (float)(1.0 / __builtin_sqrt((double)pr.hs));
  p.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)pr.hs));
  const int n_sm = device_sm_count();
  const int grid = p.n_items < n_sm ? p.n_items : n_sm;   // persistent: one CTA per SM
  const WorkDeal deal = launch_deal_bwd(pr.causal, p.n_kv, p.BH, grid);
  if (pr.hs == 64)
    e = pr.causal ? launch_bwd_main<64, true>(map_qkv, map_dout, map_dqkv, map_dqacc, p, deal, grid, stream)
                  : launch_bwd_main<64, false>(map_qkv, map_dout, map_dqkv, map_dqacc, p, deal, grid, stream);
  else
    e = pr.causal ? launch_bwd_main<32, true>(map_qkv, map_dout, map_dqkv, map_dqacc, p, deal, grid, stream)
                  : launch_bwd_main<32, false>(map_qkv, map_dout, map_dqkv, map_dqacc, p, deal, grid, stream);
  if (e != cudaSuccess) return e;

  ProfileScope ps(K_BWD_DQ, stream);
  return launch_pdl(attn_bwd_dq_out, dim3((unsigned)blocks), dim3(threads), 0, stream,
                    reinterpret_cast<const float4*>(ws_dq), static_cast<uint4*>(dqkv), pr.C, n_vec,
                    device_error_word());
}

}  // namespace attn
