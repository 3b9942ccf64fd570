// Decode forward: a few new query tokens attending to a key/value cache.
//
// In autoregressive inference ("LLM Systems 10 & 11: Accelerating Transformer
// Training and Inference", §2.2, and the `step` offset of its §1 fused
// embedding kernel, which places the new tokens after the ones already
// processed) the newest Tq tokens of each sequence attend to every key up to
// their own position.
// The layout stays llm.c's: qkv is (B, L, 3C); its K and V slots for positions
// 0..L-1 are the cache (the new tokens included), and the queries are the last
// Tq rows. Query i sits at position p_i = L - Tq + i and sees keys 0..p_i:
//   out[b,i,h*hs+d] = sum_{j<=p_i} softmax_j(scale * q_i . k_j) v_j[d]
//   lse[b,h,i]      = logsumexp_{j<=p_i}(scale * q_i . k_j)
// With Tq small the arithmetic is a few multiply-adds per byte of K and V, so
// the work is a stream over the cache, bound by HBM bandwidth (kept off the
// tensor core: reshaping it into an MMA would not move the bound):
//   attn_decode_split   one CTA per (b, h, chunk of 128 keys):
//                       the chunk's K and V rows arrive in shared memory by
//                       two bulk tensor copies issued at the start (V lands
//                       while the scores are formed); q in shared memory;
//                       every row is read by hs/8 lanes, 8 elements each;
//                       partial dot products summed across those lanes; a
//                       chunk-local softmax (max, exp2, sum); the partial
//                       output summed over the rows of a warp and the warps;
//                       written as (m, l, o)
//   attn_decode_combine one warp per (b, h, i): merges the chunks' partial
//                       results (log-sum-exp rescaling) into out, lse
#include "../../include/attn.h"
#include "common.cuh"

namespace attn {
namespace deck {

constexpr int THREADS = 128;
constexpr int MAX_TQ = 8;

struct Params {
  const void* qkv;
  void* out;
  float* lse;
  float* part;                          // [B*NH][n_split][Tq][HS + 2]: m, l, o[HS]
  int* err;
  int L, C, NH, Tq, n_split;
  int BH;                               // B * NH
  float scale_log2;
};

template <typename E>
__device__ __forceinline__ float ld_e(const E* p);
template <>
__device__ __forceinline__ float ld_e<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_e<uint16_t>(const uint16_t* p) {
  return __uint_as_float((uint32_t)(*p) << 16);
}

// Load 8 consecutive elements (16 bytes of bf16 or 2 x 16 bytes of fp32) as fp32.
template <typename E>
__device__ __forceinline__ void load8(const E* src, float (&x)[8]) {
  if constexpr (sizeof(E) == 4) {
    const float4 a = *reinterpret_cast<const float4*>(src);
    const float4 c = *reinterpret_cast<const float4*>(src + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
}

template <typename E>
struct Chunk {
  // keys per split CTA: the K and V rows of a chunk are staged in shared memory
  static constexpr int N = 128;
};

// Transposing butterfly over lane masks MASK, MASK/2, ..., MASK_LO. Each lane
// enters with N partial sums v[0..N) (the same N quantities in every lane of
// the group). At a level with CNT > 1 live values the lane keeps the half its
// lane bit selects, sends the other half to its partner and adds what it gets
// back; with one live value it does a plain butterfly add. On return v[0..)
// holds complete sums of quantities first, first + 1, ...: N / 2^levels of
// them, or one (then shared by the lanes that differ only in the plain-add bits).
template <int N, int CNT, int MASK, int MASK_LO>
struct TRed {
  static __device__ __forceinline__ void run(float (&v)[N], int lane, int& first) {
    if constexpr (CNT > 1) {
      constexpr int H = CNT / 2;
      const bool hi = (lane & MASK) != 0;
#pragma unroll
      for (int k = 0; k < H; ++k) {
        const float send = hi ? v[k] : v[k + H];
        const float keep = hi ? v[k + H] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
      }
      if (hi) first += H;
      if constexpr (MASK > MASK_LO) TRed<N, H, MASK / 2, MASK_LO>::run(v, lane, first);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], MASK);
      if constexpr (MASK > MASK_LO) TRed<N, 1, MASK / 2, MASK_LO>::run(v, lane, first);
    }
  }
};
__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// TQ: the largest Tq this instantiation serves (1, 4 or 8); its per-query
// shared arrays and accumulators are sized by it, so the common one-token step
// keeps more CTAs resident per SM.
// With bf16 inputs and several query tokens both products run on the tensor
// core. S^T = K Q^T for the chunk's 128 keys (TMEM lanes) and the queries
// padded to 16 (columns), one tcgen05 group of hs/16 instructions, read back
// one key row per thread. The exponentials go to shared memory as bf16 P,
// rows = queries, K-major in the 128-byte swizzle (one 8-row atom per 64-key
// half, the rows below Tq written; the rows past them that the M = 128
// product reads are other data, and only output rows below Tq are used), and
// O = P V is a second group (N = hs, 8 instructions, over the columns S^T
// held) whose rows warp 0 reads from TMEM. 64 TMEM columns per CTA.
// K, V and the queries arrive by swizzled tensor copies (map_kq: box
// {hs, 128 rows}, map_q: box {hs, 16 rows}). The 16 query rows sit where P
// is written later (S^T has been computed from them by then), so a CTA holds
// 2 KB + its 32 KB chunk and six CTAs fit an SM. One query token, or fp32
// inputs, keep both products on the FMA pipe (exact fp32 products).
template <typename E, int HS, int TQ>
struct DecodeMma {
  static constexpr bool on = sizeof(E) == 2 && TQ > 1;
};
constexpr int P_ROWS = 8;                       // query rows of P per key half: one swizzle atom
constexpr int P_TILE_BYTES = 2 * P_ROWS * 128;  // P: 2 key halves x 8 query rows x 128 bytes
constexpr int TMEM_COLS = 64;                   // S^T (16 columns), then O over them (hs columns)
template <typename E, int HS, int TQ>
__host__ __device__ constexpr int split_smem_bytes() {
  static_assert(!DecodeMma<E, HS, TQ>::on || (TQ <= P_ROWS && 16 * HS * 2 <= P_TILE_BYTES),
                "P rows hold every query; the 16 query rows fit where P goes");
  return DecodeMma<E, HS, TQ>::on ? P_TILE_BYTES + 2 * Chunk<E>::N * HS * (int)sizeof(E) + 1024
                                  : 2 * Chunk<E>::N * HS * (int)sizeof(E) + 128;
}

template <typename E, int HS, int TQ>
__global__ void __launch_bounds__(THREADS)
attn_decode_split(const __grid_constant__ CUtensorMap map_qkv, const __grid_constant__ CUtensorMap map_kq,
                  const __grid_constant__ CUtensorMap map_q, const Params p) {
  constexpr bool MMA = DecodeMma<E, HS, TQ>::on;
  static_assert(!MMA || THREADS == Chunk<E>::N, "tensor-core scores: one thread per key of the chunk");
  // A K or V row (HS elements) is read by LPR lanes, 8 elements each, so a
  // warp instruction covers whole rows; GROUPS rows at a time.
  constexpr int CH = Chunk<E>::N;
  constexpr int LPR = HS / 8;                 // lanes per row (8 for hs 64, 4 for hs 32)
  constexpr int GROUPS = THREADS / LPR;       // rows per CTA step
  constexpr uint32_t BYTES = CH * HS * sizeof(E);
  // scores: TQ partial dot products reduced over the LPR lanes of a row
  constexpr int S_LEVELS = ilog2(LPR);
  constexpr int S_OUT = TQ >> S_LEVELS > 0 ? (TQ >> S_LEVELS) : 1;      // sums per lane afterwards
  constexpr int S_DUP = (1 << S_LEVELS) * S_OUT / TQ;                  // lanes holding the same sum
  // outputs: TQ x 8 partial sums reduced over the rows of a warp
  constexpr int O_LEVELS = ilog2(32 / LPR);
  constexpr int O_OUT = (8 * TQ) >> O_LEVELS;
  static_assert(O_OUT >= 1, "output reduction leaves at least one value per lane");
  extern __shared__ uint8_t smem_raw[];
  // the tensor core reads swizzled tiles from 1024-byte aligned starts; P
  // comes first, so its M = 128 operand reads stay inside the allocation
  constexpr uintptr_t ALIGN = MMA ? 1023 : 127;
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + ALIGN) & ~ALIGN);
  uint8_t* sP = sbase;                          // MMA path only
  E* sK = reinterpret_cast<E*>(sbase + (MMA ? P_TILE_BYTES : 0));
  E* sV = sK + CH * HS;
  E* sQ = reinterpret_cast<E*>(sP);             // MMA path: 16 query rows, overwritten by P once S^T is done
  __shared__ float sp[MMA ? 1 : TQ][MMA ? 1 : CH];   // CUDA-core path: scores, then p
  __shared__ float red[TQ][THREADS / 32];
  __shared__ float row_m[TQ];
  __shared__ float red_l[MMA ? TQ : 1][THREADS / 32];   // tensor-core path: row sums per warp
  __shared__ float sacc[MMA ? 1 : THREADS / 32][MMA ? 1 : TQ][MMA ? 1 : HS];
  __shared__ uint64_t bar_k, bar_v, bar_s, bar_o;
  __shared__ uint32_t tmem_sh;
  __shared__ volatile int abort_sh;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x % p.n_split;
  const int bh = blockIdx.x / p.n_split;
  const int b = bh / p.NH, h = bh % p.NH;
  const int L = p.L, C = p.C, Tq = p.Tq;
  const int j0 = split * CH;
  const int nk = min(CH, L - j0);
  const int g = tid / LPR, db = (tid % LPR) * 8;   // row group, first of this lane's 8 columns
  // (b, h) of this CTA inside the batch: then every q row and record index is
  // (the same decision in every thread, taken before any barrier)
  if (!ATTN_IN_RANGE(bh < p.BH && L >= Tq && Tq <= TQ, p.err)) return;
  // the whole chunk of K and of V, one bulk tensor copy each (rows past L read
  // as zero); V lands while the scores and the softmax are computed
  if (tid == 0) {
    abort_sh = 0;
    mbar_init(&bar_k, 1);
    mbar_init(&bar_v, 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o, 1);
    fence_mbar_init();
    if constexpr (MMA) {
      // K (swizzled) and the 16 rows from the first query on (rows past L read as zero)
      mbar_arrive_expect_tx(&bar_k, BYTES + 16 * HS * 2);
      tma_load_3d(sK, &map_kq, &bar_k, C + h * HS, j0, b);
      tma_load_3d(sQ, &map_q, &bar_k, h * HS, L - Tq, b);
    } else {
      mbar_arrive_expect_tx(&bar_k, BYTES);
      tma_load_3d(sK, &map_qkv, &bar_k, C + h * HS, j0, b);
    }
    mbar_arrive_expect_tx(&bar_v, BYTES);
    tma_load_3d(sV, MMA ? &map_kq : &map_qkv, &bar_v, 2 * C + h * HS, j0, b);
  }
  if constexpr (MMA) {
    if (warp == 0) {
      tmem_alloc(&tmem_sh, TMEM_COLS);
      tmem_relinquish();
    }
  }
  // this lane's 8 columns of the queries (the last Tq positions), in registers
  float2 qr[MMA ? 1 : TQ][4];
  if constexpr (!MMA) {
    const size_t rs = (size_t)3 * C;
    const E* qbase = static_cast<const E*>(p.qkv) + (size_t)b * L * rs + h * HS + db;
#pragma unroll
    for (int i = 0; i < TQ; ++i) {
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (i < Tq) load8<E>(qbase + (size_t)(L - Tq + i) * rs, v);
#pragma unroll
      for (int k = 0; k < 4; ++k) qr[i][k] = make_float2(v[2 * k], v[2 * k + 1]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  bool ok = mbar_wait(&bar_k, 0, &abort_sh, p.err);
  using G = TileGeom<HS>;
  const uint32_t tmem = MMA ? tmem_sh : 0u;
  if constexpr (MMA) {
    if (tid == 0 && ok) {
      tc_fence_after();
      const uint64_t dk = make_sdesc(smem_u32(sK), 16, G::ATOM_BYTES, G::SWZ);
      const uint64_t dq = make_sdesc(smem_u32(sQ), 16, G::ATOM_BYTES, G::SWZ);
      constexpr uint32_t idesc = make_idesc_bf16(CH, 16, false, false);
#pragma unroll
      for (int k = 0; k < HS / 16; ++k) mma_ss(tmem, desc_add(dk, k * 32), desc_add(dq, k * 32), idesc, k > 0);
      mma_commit(&bar_s);
    }
    ok = mbar_wait(&bar_s, 0, &abort_sh, p.err) && ok;
    // this thread's key j: its scaled scores for the Tq queries (log2 units)
    const int j = tid;                                // key of this thread = TMEM lane
    float xs[TQ];
#pragma unroll
    for (int i = 0; i < TQ; ++i) xs[i] = -INFINITY;
    if (ok) {
      tc_fence_after();
      uint32_t sc[16];
      tmem_ld16_wait(tmem + ((uint32_t)(warp * 32) << 16), sc);
#pragma unroll
      for (int i = 0; i < TQ; ++i)
        if (i < Tq && j < nk && j0 + j <= L - Tq + i) xs[i] = __uint_as_float(sc[i]) * p.scale_log2;
    }
    tc_fence_before();                              // S^T read: O may overwrite its columns
    // chunk-local softmax per query from registers: warp maxima, then the
    // four warps' through red; exponentials as bf16 P; warp sums into red_l
#pragma unroll
    for (int i = 0; i < TQ; ++i) {
      if (i < Tq) {
        float m = xs[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) red[i][warp] = m;
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < TQ; ++i) {
      if (i < Tq) {
        float m = red[i][0];
#pragma unroll
        for (int w = 1; w < THREADS / 32; ++w) m = fmaxf(m, red[i][w]);
        const float e = m == -INFINITY ? 0.f : ex2_approx(xs[i] - m);
        // P[i][j] (bf16) at row i of key half j/64, chunk (j%64)/8 swizzled by row
        const int kk = j & 63;
        *reinterpret_cast<uint16_t*>(sP + (j >> 6) * (P_ROWS * 128) + i * 128 + ((((kk >> 3) ^ (i & 7)) << 4)) +
                                     (kk & 7) * 2) = (uint16_t)(pack_bf16x2(e, 0.f) & 0xFFFFu);
        float l = e;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) red_l[i][warp] = l;
        if (tid == i) row_m[i] = m;
      }
    }
    fence_proxy_async_smem();                         // P is read by the tensor core
    __syncthreads();
    ok = mbar_wait(&bar_v, 0, &abort_sh, p.err) && ok;
    // O = P V: A = P (K-major, the second key half one atom on), B = V (MN-major)
    if (tid == 0 && ok) {
      tc_fence_after();
      const uint64_t dp = make_sdesc(smem_u32(sP), 16, 1024, SWZ_128B);
      const uint64_t dv = make_sdesc(smem_u32(sV), 16, G::ATOM_BYTES, G::SWZ);
      constexpr uint32_t idesc = make_idesc_bf16(CH, HS, false, true);
#pragma unroll
      for (int k = 0; k < CH / 16; ++k)
        mma_ss(tmem, desc_add(dp, (k >> 2) * (P_ROWS * 128) + (k & 3) * 32),
               desc_add(dv, k * 16 * G::ROW_BYTES), idesc, k > 0);
      mma_commit(&bar_o);
    }
    ok = mbar_wait(&bar_o, 0, &abort_sh, p.err) && ok;
    if (warp == 0 && ok) {
      // query rows = TMEM lanes 0..Tq-1: m (log2 units), l, o[HS]
      tc_fence_after();
      uint32_t o[HS];
#pragma unroll
      for (int c0 = 0; c0 < HS; c0 += 16) {
        uint32_t t16[16];
        tmem_ld16_wait(tmem + c0, t16);
#pragma unroll
        for (int k = 0; k < 16; ++k) o[c0 + k] = t16[k];
      }
      if (lane < Tq) {
        float* rec = p.part + (((size_t)bh * p.n_split + split) * Tq + lane) * (HS + 2);
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < THREADS / 32; ++w) l += red_l[lane][w];
        rec[0] = row_m[lane];
        rec[1] = l;
        // records are HS + 2 floats long: 8-byte aligned, so pairs
#pragma unroll
        for (int d = 0; d < HS; d += 2)
          *reinterpret_cast<float2*>(rec + 2 + d) = make_float2(__uint_as_float(o[d]), __uint_as_float(o[d + 1]));
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      // a wait that gave up may leave a group in flight: let it land first
      if (abort_sh)
        for (int k = 0; k < 1000; ++k) __nanosleep(1000);
      __syncwarp();
      tmem_dealloc(tmem, TMEM_COLS);
    }
    return;
  } else
  // scores: packed partial dot products over the lane's 8 columns, then the
  // transposing butterfly over the row's lanes
  for (int r0 = 0; r0 < CH; r0 += GROUPS) {
    const int j = r0 + g;
    float kv[8];
    load8<E>(sK + j * HS + db, kv);
    float part[TQ];
#pragma unroll
    for (int i = 0; i < TQ; ++i) {
      float2 a = mul2(qr[i][0], make_float2(kv[0], kv[1]));
      a = fma2(qr[i][1], make_float2(kv[2], kv[3]), a);
      a = fma2(qr[i][2], make_float2(kv[4], kv[5]), a);
      a = fma2(qr[i][3], make_float2(kv[6], kv[7]), a);
      part[i] = a.x + a.y;
    }
    int first = 0;
    if constexpr (S_LEVELS > 0) TRed<TQ, TQ, LPR / 2, 1>::run(part, lane, first);
    if ((lane & (S_DUP - 1)) == 0) {
#pragma unroll
      for (int k = 0; k < S_OUT; ++k) {
        const int i = first + k;
        if (i < Tq) sp[i][j] = (j < nk && j0 + j <= L - Tq + i) ? part[k] * p.scale_log2 : -INFINITY;   // log2 units
      }
    }
  }
  __syncthreads();
  // chunk-local softmax per query: max, then exp2 and sum
  for (int i = 0; i < Tq; ++i) {
    float m = -INFINITY;
    for (int j = tid; j < CH; j += THREADS) m = fmaxf(m, sp[i][j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[i][warp] = m;
  }
  __syncthreads();
  if (tid < Tq) {
    float m = red[tid][0];
#pragma unroll
    for (int w = 1; w < THREADS / 32; ++w) m = fmaxf(m, red[tid][w]);
    row_m[tid] = m;
  }
  __syncthreads();
  for (int i = 0; i < Tq; ++i) {
    const float m = row_m[i];
    float l = 0.f;
    for (int j = tid; j < CH; j += THREADS) {
      const float e = m == -INFINITY ? 0.f : ex2_approx(sp[i][j] - m);
      sp[i][j] = e;
      l += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) red[i][warp] = l;
  }
  __syncthreads();
  ok = mbar_wait(&bar_v, 0, &abort_sh, p.err) && ok;
  // partial outputs: each lane accumulates its 8 columns over its rows of the
  // chunk for every query (packed pairs), then the transposing butterfly sums
  // the rows of the warp and the warps are summed through shared memory
  float2 acc[TQ][4];
#pragma unroll
  for (int i = 0; i < TQ; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[i][k] = make_float2(0.f, 0.f);
#pragma unroll 4
  for (int r0 = 0; r0 < CH; r0 += GROUPS) {
    const int j = r0 + g;
    float vv[8];
    load8<E>(sV + j * HS + db, vv);               // rows past L are zero, their p is 0
#pragma unroll
    for (int i = 0; i < TQ; ++i) {
      if (i < Tq) {
        const float pj = sp[i][j];
        const float2 p2 = make_float2(pj, pj);
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[i][k] = fma2(p2, make_float2(vv[2 * k], vv[2 * k + 1]), acc[i][k]);
      }
    }
  }
  {
    float o[8 * TQ];
#pragma unroll
    for (int i = 0; i < TQ; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        o[i * 8 + 2 * k] = acc[i][k].x;
        o[i * 8 + 2 * k + 1] = acc[i][k].y;
      }
    int first = 0;
    TRed<8 * TQ, 8 * TQ, 16, LPR>::run(o, lane, first);
#pragma unroll
    for (int k = 0; k < O_OUT; ++k) {
      const int idx = first + k, i = idx / 8, dd = idx % 8;
      if (i < Tq) sacc[warp][i][db + dd] = o[k];
    }
  }
  __syncthreads();
  if (!ok) return;                                  // the error word says why
  // partial record: m (log2 units), l, o[HS]
  float* rec = p.part + ((size_t)bh * p.n_split + split) * Tq * (HS + 2);
  for (int x = tid; x < Tq * HS; x += THREADS) {
    const int i = x / HS, d = x % HS;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) o += sacc[w][i][d];
    rec[i * (HS + 2) + 2 + d] = o;
  }
  if (tid < Tq) {
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) l += red[tid][w];
    rec[tid * (HS + 2) + 0] = row_m[tid];
    rec[tid * (HS + 2) + 1] = l;
  }
}

// One warp per (b, h, query), four per block: merge the chunks' partials.
// PER_LANE (up to four query tokens): each lane takes every 32nd chunk record
// (all of a record's loads are independent, so the set is fetched in about one
// round trip), sums its records' outputs weighted by 2^(m_s - M), and a
// transposing butterfly over the lanes leaves columns 2*lane, 2*lane+1 (hs 64)
// or lane (hs 32) in each lane. Otherwise (five to eight queries, more warps
// than the GPU holds at once) the warp walks the records in order, hs/32
// columns per lane and four records' loads in flight, so every load is a whole
// record row.
constexpr int COMBINE_WARPS = 4;
template <typename E, int HS, bool PER_LANE>
__global__ void __launch_bounds__(32 * COMBINE_WARPS) attn_decode_combine(const Params p) {
  constexpr int DPL = HS / 32;                       // output columns per lane
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * COMBINE_WARPS + (threadIdx.x >> 5);
  const int Tq = p.Tq;
  if (gw >= p.BH * Tq) return;
  const int i = gw % Tq, bh = gw / Tq;
  const int b = bh / p.NH, h = bh % p.NH;
  // only chunks that hold a visible key of this query contribute
  const int n = (p.L - Tq + i) / Chunk<E>::N + 1;
  if (!ATTN_IN_RANGE(n <= p.n_split, p.err)) return;
  const size_t stride = (size_t)Tq * (HS + 2);       // floats between two chunks' records
  const float* rec = p.part + (size_t)bh * p.n_split * stride + (size_t)i * (HS + 2);
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, rec[s * stride]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if constexpr (!PER_LANE) {
    float l = 0.f;
    for (int s = lane; s < n; s += 32) l = fmaf(rec[s * stride + 1], ex2_approx(rec[s * stride] - M), l);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    float acc[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[k] = 0.f;
    int s = 0;
    for (; s + 4 <= n; s += 4) {
      float w[4], v[4][DPL];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float* r = rec + (s + u) * stride;
        w[u] = r[0];
#pragma unroll
        for (int k = 0; k < DPL; ++k) v[u][k] = r[2 + k * 32 + lane];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float wu = ex2_approx(w[u] - M);
#pragma unroll
        for (int k = 0; k < DPL; ++k) acc[k] = fmaf(v[u][k], wu, acc[k]);
      }
    }
    for (; s < n; ++s) {
      const float* r = rec + s * stride;
      const float wu = ex2_approx(r[0] - M);
#pragma unroll
      for (int k = 0; k < DPL; ++k) acc[k] = fmaf(r[2 + k * 32 + lane], wu, acc[k]);
    }
    const float inv_l = 1.f / l;
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
      const float val = acc[k] * inv_l;
      const size_t oi = ((size_t)b * Tq + i) * p.C + h * HS + k * 32 + lane;
      if constexpr (sizeof(E) == 4) static_cast<float*>(p.out)[oi] = val;
      else static_cast<uint16_t*>(p.out)[oi] = (uint16_t)(pack_bf16x2(val, 0.f) & 0xFFFFu);
    }
    if (lane == 0) p.lse[(size_t)bh * Tq + i] = (M + __log2f(l)) * 0.69314718055994531f;
  } else {
    float acc[HS];
#pragma unroll
    for (int d = 0; d < HS; ++d) acc[d] = 0.f;
    float l = 0.f;
    for (int s = lane; s < n; s += 32) {
      const float* r = rec + s * stride;
      float v[HS];
#pragma unroll
      for (int d = 0; d < HS; d += 2) {                // records are 8-byte aligned
        const float2 x = *reinterpret_cast<const float2*>(r + 2 + d);
        v[d] = x.x;
        v[d + 1] = x.y;
      }
      const float w = ex2_approx(r[0] - M);
      l = fmaf(r[1], w, l);
#pragma unroll
      for (int d = 0; d < HS; ++d) acc[d] = fmaf(v[d], w, acc[d]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    int first = 0;
    TRed<HS, HS, 16, 1>::run(acc, lane, first);        // acc[0..DPL): columns first, first+1, ...
    const float inv_l = 1.f / l;
    const size_t oi = ((size_t)b * Tq + i) * p.C + h * HS + first;
    if constexpr (DPL == 2) {
      if constexpr (sizeof(E) == 4)
        *reinterpret_cast<float2*>(static_cast<float*>(p.out) + oi) = make_float2(acc[0] * inv_l, acc[1] * inv_l);
      else
        *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + oi) = pack_bf16x2(acc[0] * inv_l, acc[1] * inv_l);
    } else {
      if constexpr (sizeof(E) == 4) static_cast<float*>(p.out)[oi] = acc[0] * inv_l;
      else static_cast<uint16_t*>(p.out)[oi] = (uint16_t)(pack_bf16x2(acc[0] * inv_l, 0.f) & 0xFFFFu);
    }
    if (lane == 0) p.lse[(size_t)bh * Tq + i] = (M + __log2f(l)) * 0.69314718055994531f;
  }
}

template <typename E, int HS>
static cudaError_t launch_t(const CUtensorMap& m, const CUtensorMap& mkq, const CUtensorMap& mq, const Params& p,
                            int BH, cudaStream_t s) {
  auto k = p.Tq == 1 ? attn_decode_split<E, HS, 1>
                     : (p.Tq <= 4 ? attn_decode_split<E, HS, 4> : attn_decode_split<E, HS, MAX_TQ>);
  const int smem = p.Tq == 1 ? split_smem_bytes<E, HS, 1>()
                             : (p.Tq <= 4 ? split_smem_bytes<E, HS, 4>() : split_smem_bytes<E, HS, MAX_TQ>());
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<(unsigned)(BH * p.n_split), THREADS, smem, s>>>(m, mkq, mq, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto c = p.Tq <= 4 ? attn_decode_combine<E, HS, true> : attn_decode_combine<E, HS, false>;
  c<<<(unsigned)((BH * p.Tq + COMBINE_WARPS - 1) / COMBINE_WARPS), 32 * COMBINE_WARPS, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace deck

int decode_chunk(bool f32) { return f32 ? deck::Chunk<float>::N : deck::Chunk<uint16_t>::N; }

size_t decode_workspace_bytes(int B, int L, int C, int NH, int Tq, bool f32) {
  const int hs = C / NH;
  const size_t n_split = (size_t)(L + decode_chunk(f32) - 1) / decode_chunk(f32);
  return (size_t)B * NH * n_split * Tq * (hs + 2) * 4;
}

int decode_max_tq() { return deck::MAX_TQ; }

// map_qkv: qkv as {3C, L, B}, box {hs, chunk rows, 1}, no swizzle; map_kq and
// map_q: the same tensor in the hs-row swizzle (128 bytes for hs 64, 64 for
// hs 32), boxes {hs, 128, 1} and {hs, 16, 1} (bf16 only; unused for fp32)
cudaError_t launch_decode(const CUtensorMap& map_qkv, const CUtensorMap& map_kq, const CUtensorMap& map_q,
                          const void* qkv, void* out, float* lse, float* part, bool f32, int B, int L, int C, int NH,
                          int Tq, cudaStream_t stream) {
  deck::Params p;
  p.qkv = qkv;
  p.out = out;
  p.lse = lse;
  p.part = part;
  p.err = device_error_word();
  p.L = L;
  p.C = C;
  p.NH = NH;
  p.Tq = Tq;
  p.n_split = (L + decode_chunk(f32) - 1) / decode_chunk(f32);
  p.BH = B * NH;
  const int hs = C / NH;
  p.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)hs));
  const int BH = B * NH;
  if (f32)
    return hs == 64 ? deck::launch_t<float, 64>(map_qkv, map_kq, map_q, p, BH, stream)
                    : deck::launch_t<float, 32>(map_qkv, map_kq, map_q, p, BH, stream);
  return hs == 64 ? deck::launch_t<uint16_t, 64>(map_qkv, map_kq, map_q, p, BH, stream)
                  : deck::launch_t<uint16_t, 32>(map_qkv, map_kq, map_q, p, BH, stream);
}

}  // namespace attn
