// backward.cu -- attention backward: dQ, dK, dV for O = softmax(scale * Q K^T) V.
//
// What it computes ("Attention kernel chains", "What the backward pass saves"):
// the forward keeps Q, K, V, O and one log-sum-exp per query row; the backward
// rebuilds each probability tile on chip as P = exp(S - LSE) and needs one more
// vector, D = rowsum(dO * O), formed once before the main loops. With
// S = scale * Q K^T, the chain rule through O = P V and P = softmax(S) gives
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q,
// a KV head's dK, dV summing over the query heads of its group; masked scores
// (bottom-right causal mask) have P = 0.
//
// How (GB300-specific): two launches.
//   * bwd_rowsum_kernel: per query row, -D and the negated base-2 LSE into a small
//     workspace (HBM-bound, tiny); the main grid launches as its programmatic
//     dependent.
//   * bwd_kernel: the dK/dV pass and the dQ pass as the two halves of one grid,
//     the dQ CTAs filling the last wave of the dK/dV ones.
//     - dK/dV (bwd_dkdv_cta): one 128-key tile per CTA looping over the query tiles
//       (a GQA group's heads stacked as rows, as in the forward). S^T = K Q^T and
//       dP^T = V dO^T in TMEM (rows = keys); eight warps write P^T in bf16 to a
//       swizzled shared-memory tile (so S^T of the next tile can overwrite S^T as
//       soon as it has been read) and dS^T in bf16 over dP^T's columns; dV += P^T dO
//       reads P^T from shared memory, dK += dS^T Q reads dS^T from TMEM, with dO and
//       Q as MN-major operands from shared memory. dK and dV accumulate in TMEM over
//       all query tiles and all heads of the group.
//     - dQ (bwd_dq_cta): one 128-row query tile per CTA looping over 128-key tiles.
//       S = Q K^T and dP = dO V^T in TMEM; the warps form dS = P * (dP - D) in bf16
//       over dP's columns; dQ += dS K takes dS straight from TMEM as the A operand.
//     The streamed tiles (Q and dO, or K and V) rotate through four shared-memory
//     slots so that the tile needed first in step j + 2 loads as soon as the step
//     j tile that is released early frees its slot.
// Computing dQ in its own pass (recomputing S and dP there) keeps every
// accumulator in TMEM and needs no atomics. MMAs of neighbouring tiles overlap
// each tile's elementwise work.
#include "common.cuh"

namespace fa {

// ---------------------------------------------------------------------------
// Per query row, into the row-vector workspace [2][B*Hq][T_pad]: -D = -rowsum(dO * O)
// (plane 0) and -lse * log2(e), the row's LSE in base 2 negated (plane 1; -inf for
// a row with no visible key, so that its P is 0). A group of d / 16 lanes takes a
// row, 32 bytes of O and of dO per lane in four 16-byte loads issued together
// (HBM-bound: every byte of O and dO is read once). The kernel launches as a
// programmatic dependent of the launch before it on the stream (for a training loop,
// the previous backward's main grid) and waits before it reads anything; every block
// lets the main kernel launch as its own programmatic dependent at once, and that
// kernel waits (griddepcontrol.wait) only where it reads these values.
__global__ void __launch_bounds__(256) bwd_rowsum_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ d_o,
                                                         const float* __restrict__ lse, float* __restrict__ vecs,
                                                         long long rows, int T, int T_pad, int d) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the work ahead on the stream is complete
  const int lanes = d / 16;  // 8 (d = 128) or 4 (d = 64): a power of two dividing 32
  const int sub = threadIdx.x & (lanes - 1);
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / lanes;
  float acc = 0.f;
  if (row < rows) {
    const uint4* pa = reinterpret_cast<const uint4*>(o + row * d + sub * 16);
    const uint4* pg = reinterpret_cast<const uint4*>(d_o + row * d + sub * 16);
    // streaming loads: this pass reads each byte once
    uint4 a[2], g[2];
    a[0] = __ldcs(pa);
    a[1] = __ldcs(pa + 1);
    g[0] = __ldcs(pg);
    g[1] = __ldcs(pg + 1);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[h]);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g[h]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = __bfloat1622float2(a2[k]);
        const float2 y = __bfloat1622float2(g2[k]);
        acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
      }
    }
  }
  for (int off = lanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sub == 0) {
    const long long bh = row / T;
    const long long at = bh * T_pad + (row - bh * T);
    const long long plane = (rows / T) * T_pad;
    const float l = lse[row];
    vecs[at] = -acc;
    vecs[plane + at] = l == -INFINITY ? -INFINITY : -l * kLog2e;
  }
}

// ---------------------------------------------------------------------------
// Shared configuration
// ---------------------------------------------------------------------------
template <int D>
struct BwCfg {
  static constexpr int BM = 128;                 // rows of a tile (TMEM lanes)
  static constexpr int BN = 128;                 // columns of S (keys, or queries for S^T)
  static constexpr int KCH = D / 64;             // 128-byte chunks along d
  static constexpr int CHUNK_BYTES = 128 * 128;  // one 128-row x 128-byte swizzled chunk
  static constexpr int TILE_BYTES = 128 * D * 2; // one 128-row tile of Q, dO, K or V
  static constexpr int STAGES = 2;
  // smem: two fixed tiles (Q and dO, or K and V), then a ring of STAGES tile pairs
  static constexpr int OFF_FIX = 0;
  static constexpr int OFF_RING = 2 * TILE_BYTES;
  // dK/dV: P^T of the current step in bf16 (128 keys x 128 queries, two 128-byte-swizzled
  // chunks of 64 queries), the A operand of dV
  static constexpr int OFF_PT = OFF_RING + STAGES * 2 * TILE_BYTES;
  static constexpr int PT_BYTES = 128 * 128 * 2;
  static constexpr int OFF_BAR = OFF_PT + PT_BYTES;
  static constexpr int OFF_VEC = OFF_BAR + 256;  // dK/dV: per ring stage, -lse2 and -D of the query columns
  // the dynamic shared memory is declared 1024-byte aligned (checked at run time): no slack
  static constexpr int SMEM = OFF_VEC + 2 * 2 * BM * 4;
  // warps 0-7 elementwise: warp w takes TMEM lanes 32(w%4).. and column half w/4
  // (every element is independent, so a pair splits a row's columns with no
  // exchange); warp 8 producer, warp 9 MMA
  static constexpr int THREADS = 320;
  static constexpr int EW_THREADS = 256;
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
  static constexpr int TMEM_COLS = 512;
  static constexpr int COL_S = 0;                // S (or S^T): fp32; P / dS (bf16) later over it
  static constexpr int COL_DP = 128;             // dP (or dP^T)
  static constexpr int COL_ACC = 256;            // dQ, or dV then dK
  // dQ: Q and dO (fixed for the whole tile) packed bf16 in TMEM, the A operands of S
  // and dP, so that those products read only their B operand from shared memory
  static constexpr int COL_QA = 384;
  static constexpr int COL_DOA = 448;
  // Packed bf16 operands (two per 32-bit column) written by column half hf over
  // the first 32 of its own 64 fp32 columns: the 16 keys (or queries) of MMA
  // K-step kk sit at column packed_col(kk) of the S (or dP) region.
  static __device__ __forceinline__ uint32_t packed_col(int kk) { return 64 * (kk >> 2) + (kk & 3) * 8; }
};

static_assert(BwCfg<128>::SMEM <= 232448, "shared memory of the d = 128 backward");

struct BwParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* neg_d;  // -D per query row, [B*Hq][T_pad]
  const float* nl2;    // -lse * log2(e) per query row (-inf: no visible key), [B*Hq][T_pad]
  int T_pad;           // T rounded up to a multiple of 4 (16-byte rows for TMA)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int B, Hq, Hkv, T, S;
  int g, rows_per_head, n_qtiles, n_ktiles;
  int causal;
  float scale;
  float c;  // scale * log2(e)
  unsigned* err;
  unsigned long long timeout_ns;
};

struct BwBars {
  uint64_t fix_full;      // the fixed tile pair landed
  uint64_t s_full;        // S (or S^T) of this step is in TMEM
  uint64_t dp_full;       // dP (or dP^T) of this step is in TMEM
  uint64_t e_first;       // dQ: S read out of TMEM; dK/dV: P^T written (even steps)
  uint64_t e_first_odd;   // dK/dV: P^T of odd steps (the warps may finish step i+1's P before
                          // the MMA warp has seen step i's)
  uint64_t s_read;        // dK/dV: S^T read out of TMEM (S^T of the next step may overwrite it)
  uint64_t pt_free;       // dK/dV: dV has read P^T from shared memory
  uint64_t e_second;      // dS (or dS^T) written
  uint64_t a_ready;       // dQ: Q and dO copied into TMEM (the A operands of S and dP)
  uint64_t acc_done;      // the last accumulation finished
  uint64_t slot_full[4];  // a streamed tile landed in ring slot t
  uint64_t slot_empty[4]; // the last MMA reading slot t finished
  uint32_t tmem_base;
  int abort_flag;
};

// Row r of a stacked 128-row query tile qt: head h_local = r / rows_per_head of
// the group, position qt * rows_per_head + r % rows_per_head.
__device__ __forceinline__ void bw_row(const BwParams& p, int qt, int r, int& h_local, int& pos) {
  h_local = r / p.rows_per_head;
  pos = qt * p.rows_per_head + (r % p.rows_per_head);
}

// The ring of both kernels: four tile slots. Step j's two streamed tiles use the
// two slots of pair j & 1, swapped every other use: the tile whose last reader comes
// late in the step (K in the dQ kernel, read by dQ; Q in the dK/dV kernel, read by
// dK) lands in the slot that the other tile of step j - 2 (V, read last by dP; dO,
// read last by dV) gave back early.
__device__ __forceinline__ int slot_late(int j) { return 2 * (j & 1) + ((j >> 1) & 1); }
__device__ __forceinline__ int slot_early(int j) { return 2 * (j & 1) + 1 - ((j >> 1) & 1); }

// ---------------------------------------------------------------------------
// dQ: one stacked query tile qt of (batch, KV head) bkv per CTA, looping over key tiles
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void bwd_dq_cta(const CUtensorMap& tmQ, const CUtensorMap& tmDO, const CUtensorMap& tmK,
                                           const CUtensorMap& tmV, const BwParams& p, const int qt,
                                           const int bkv) {
  using C = BwCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  uint8_t* sQ = smem + C::OFF_FIX;
  uint8_t* sDO = sQ + C::TILE_BYTES;
  uint8_t* sRing = smem + C::OFF_RING;  // four tile slots (slot_late / slot_early) for K and V
  BwBars* bars = reinterpret_cast<BwBars*>(smem + C::OFF_BAR);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = bkv / p.Hkv;
  const int kvh = bkv % p.Hkv;
  const int shift = p.S - p.T;
  // key tiles this query tile needs: causal stops at the last row's diagonal
  int kv_end = p.S;
  if (p.causal) kv_end = min(p.S, min((qt + 1) * p.rows_per_head, p.T) - 1 + shift + 1);
  const int nj = kv_end > 0 ? (kv_end + C::BN - 1) / C::BN : 0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->fix_full, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->e_first, C::EW_THREADS);
    mbar_init(&bars->e_second, C::EW_THREADS);
    mbar_init(&bars->a_ready, C::EW_THREADS);
    mbar_init(&bars->acc_done, 1);
    for (int t = 0; t < 4; ++t) {
      mbar_init(&bars->slot_full[t], 1);
      mbar_init(&bars->slot_empty[t], 1);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::MMA_WARP) tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;
  const uint64_t tmo = p.timeout_ns;
  const uint64_t tmo_unwind = unwind_timeout(tmo);  // copies landing, MMAs draining
  auto fail = [&](unsigned site) {
    record_error(p.err, FA_ERR_TIMEOUT, site);
    *abort_flag = 1;
  };

  if (warp == C::PRODUCER_WARP) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars->fix_full, 2 * C::TILE_BYTES);
      for (int c = 0; c < C::KCH; ++c) {
        tma_load_4d(sQ + c * C::CHUNK_BYTES, &tmQ, &bars->fix_full, c * 64, qt * p.rows_per_head, kvh * p.g, b);
        tma_load_4d(sDO + c * C::CHUNK_BYTES, &tmDO, &bars->fix_full, c * 64, qt * p.rows_per_head, kvh * p.g, b);
      }
      int issued = 0;  // tiles whose K and V loads were both issued
      int k_only = -1;  // a tile whose K load was issued alone
      for (int j = 0; j < nj; ++j) {
        // each slot's previous use was key tile j - 2
        const int ks = slot_late(j), vs = slot_early(j);
        const uint32_t prev = ((j >> 1) - 1) & 1;
        if (j >= 2 && !mbar_wait(&bars->slot_empty[ks], prev, tmo, abort_flag)) {
          fail(SITE_BW_PRODUCER);
          break;
        }
        mbar_arrive_expect_tx(&bars->slot_full[ks], C::TILE_BYTES);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(sRing + ks * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmK, &bars->slot_full[ks], c * 64,
                      j * C::BN, bkv);
        k_only = j;
        if (j >= 2 && !mbar_wait(&bars->slot_empty[vs], prev, tmo, abort_flag)) {
          fail(SITE_BW_PRODUCER);
          break;
        }
        mbar_arrive_expect_tx(&bars->slot_full[vs], C::TILE_BYTES);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(sRing + vs * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmV, &bars->slot_full[vs], c * 64,
                      j * C::BN, bkv);
        k_only = -1;
        issued = j + 1;
      }
      if (*abort_flag) {
        // copies in flight must land before the CTA exits
        mbar_wait(&bars->fix_full, 0, tmo_unwind);
        for (int x = max(0, issued - 2); x < issued; ++x) {
          mbar_wait(&bars->slot_full[slot_late(x)], (x >> 1) & 1, tmo_unwind);
          mbar_wait(&bars->slot_full[slot_early(x)], (x >> 1) & 1, tmo_unwind);
        }
        if (k_only >= 0) mbar_wait(&bars->slot_full[slot_late(k_only)], (k_only >> 1) & 1, tmo_unwind);
      }
    }
  } else if (warp == C::MMA_WARP) {
    const bool leader = elect_one();
    constexpr uint32_t idesc_ss = idesc_bf16_f32(128, C::BN, 0, 0);  // S, dP: A from TMEM, B K-major
    constexpr uint32_t idesc_ts = idesc_bf16_f32(128, D, 0, 1);      // dQ: A from TMEM, B MN-major
    const uint64_t dRing = smem_desc_sw128(smem_u32(sRing), 16, 1024);                    // K (for S), V (for dP)
    const uint64_t dRingKmn = smem_desc_sw128(smem_u32(sRing), C::CHUNK_BYTES, 1024);     // K as the B of dQ
    auto slot_off = [](int t) { return static_cast<uint64_t>((t * C::TILE_BYTES) >> 4); };
    // Issue order: S(0), dP(0), then per key tile j: S(j+1) (once the warps have read
    // S(j) out), dQ(j) += dS(j) K_j (dS over dP's columns), dP(j+1) (after dQ(j) in
    // issue order, so it never overwrites dS(j) before it is read). The MMAs of the
    // neighbouring tiles run while the warps work on tile j. S and dP take Q and dO
    // from TMEM (16 d-values = 8 packed columns per K step): every product reads only
    // its B operand (K or V) from shared memory.
    auto issue_s = [&](int j) {
      const uint64_t so = slot_off(slot_late(j));
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4);
          tc_mma_ts(tmem + C::COL_S, tmem + C::COL_QA + kk * 8, dRing + so + off, idesc_ss, kk > 0 ? 1u : 0u);
        }
        tc_commit(&bars->s_full);
      }
    };
    // dP(j); V(j)'s slot is free once it completes
    auto issue_dp = [&](int j) {
      const int vs = slot_early(j);
      const uint64_t so = slot_off(vs);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4);
          tc_mma_ts(tmem + C::COL_DP, tmem + C::COL_DOA + kk * 8, dRing + so + off, idesc_ss, kk > 0 ? 1u : 0u);
        }
        tc_commit(&bars->dp_full);
        tc_commit(&bars->slot_empty[vs]);
      }
    };
    // Q and dO reach TMEM through the elementwise warps (after fix_full)
    bool ok = mbar_wait(&bars->a_ready, 0, tmo, abort_flag);
    if (ok && nj > 0) {
      ok = mbar_wait(&bars->slot_full[slot_late(0)], 0, tmo, abort_flag) &&
           mbar_wait(&bars->slot_full[slot_early(0)], 0, tmo, abort_flag);
      tc_fence_after();
      if (ok) {
        issue_s(0);
        issue_dp(0);
      }
    }
    for (int j = 0; ok && j < nj; ++j) {
      const uint32_t use_next = ((j + 1) >> 1) & 1;  // slot parity of key tile j + 1
      if (j + 1 < nj) {
        // S(j+1) overwrites S(j): the warps must have read it out
        if (!mbar_wait(&bars->e_first, j & 1, tmo, abort_flag) ||
            !mbar_wait(&bars->slot_full[slot_late(j + 1)], use_next, tmo, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(j + 1);
      }
      if (!mbar_wait(&bars->e_second, j & 1, tmo, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int ks = slot_late(j);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          tc_mma_ts(tmem + C::COL_ACC, tmem + C::COL_DP + C::packed_col(kk),
                    dRingKmn + slot_off(ks) + static_cast<uint64_t>((kk * 2048) >> 4), idesc_ts,
                    (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&bars->slot_empty[ks]);
      }
      if (j + 1 < nj) {
        if (!mbar_wait(&bars->slot_full[slot_early(j + 1)], use_next, tmo, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_dp(j + 1);
      }
    }
    if (!ok && leader) fail(SITE_BW_MMA);
    if (leader) tc_commit(&bars->acc_done);
    mbar_wait(&bars->acc_done, 0, tmo_unwind);
  } else {
    // ---- elementwise warps: one query row per thread pair (TMEM lane), column half hf
    const int r = threadIdx.x & 127;
    const int hf = warp >> 2;
    int h_local, pos;
    bw_row(p, qt, r, h_local, pos);
    const bool row_valid = pos < p.T;
    const int h = kvh * p.g + h_local;
    const size_t row_index = (static_cast<size_t>(b) * p.Hq + h) * p.T + (row_valid ? pos : 0);
    // P = 2^(S*c - lse*log2e); rows past T and rows with no visible key get P = 0
    const size_t vi = (static_cast<size_t>(b) * p.Hq + h) * p.T_pad + (row_valid ? pos : 0);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the row pass's values are complete and visible
    const float nl2_row = row_valid ? __ldg(p.nl2 + vi) : -INFINITY;
    const float nd_row = row_valid ? __ldg(p.neg_d + vi) : 0.f;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::COL_S;
    const uint32_t tDP = tmem + lane_base + C::COL_DP;
    const float2 c2 = make_float2(p.c, p.c);
    const float2 nl2 = make_float2(nl2_row, nl2_row);
    const float2 nd2 = make_float2(nd_row, nd_row);
    // Q and dO rows into TMEM as packed bf16 pairs (column c holds d-values 2c, 2c+1):
    // row r of the 128-byte-swizzled smem tiles, this column half's D/4 columns
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->fix_full, 0, tmo, abort_flag));
    if (ok) {
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint8_t* src = which ? sDO : sQ;
        uint32_t wv[D / 4];
        // d = 128: half hf is chunk hf (64 values); d = 64: half hf is units 4hf..4hf+3 of the one chunk
#pragma unroll
        for (int u = 0; u < D / 16; ++u) {
          const int unit = D == 128 ? u : 4 * hf + u;
          const uint8_t* rowp = src + (D == 128 ? hf * C::CHUNK_BYTES : 0) + r * 128;
          const uint4 x = *reinterpret_cast<const uint4*>(rowp + ((unit ^ (r & 7)) << 4));
          wv[4 * u + 0] = x.x;
          wv[4 * u + 1] = x.y;
          wv[4 * u + 2] = x.z;
          wv[4 * u + 3] = x.w;
        }
        const uint32_t col = (which ? C::COL_DOA : C::COL_QA) + hf * (D / 4);
        if constexpr (D == 128) {
          tmem_st32(tmem + lane_base + col, wv);
        } else {
          tmem_st16(tmem + lane_base + col, wv);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->a_ready);
    }
    for (int j = 0; ok && j < nj; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full, j & 1, tmo, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int key0 = j * C::BN + hf * 64;
      // last visible key of this row (bottom-right causal), relative to this half's first key
      const int lim = (p.causal ? min(p.S - 1, pos + shift) : p.S - 1) - key0;
      // P = 2^(S*c - lse2) for this half's 64 keys, kept in registers; S is then free
      float pv[64];
      {
        uint32_t sr[2][32];
        tmem_ld32(tS + hf * 64, sr[0]);
        tmem_ld32(tS + hf * 64 + 32, sr[1]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bars->e_first);
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float2 x = ffma2(make_float2(__uint_as_float(sr[i >> 5][i & 31]), __uint_as_float(sr[i >> 5][(i & 31) + 1])),
                                 c2, nl2);
          pv[i] = ex2_approx(x.x);
          pv[i + 1] = ex2_approx(x.y);
        }
        if (__any_sync(0xffffffffu, lim < 63)) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i > lim) pv[i] = 0.f;
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->dp_full, j & 1, tmo, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        uint32_t dr[2][32];
        tmem_ld32(tDP + hf * 64, dr[0]);
        tmem_ld32(tDP + hf * 64 + 32, dr[1]);
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int e = cc * 32 + 2 * i;
            const float2 t = fadd2(make_float2(__uint_as_float(dr[cc][2 * i]), __uint_as_float(dr[cc][2 * i + 1])), nd2);
            const float2 g2 = fmul2(make_float2(pv[e], pv[e + 1]), t);
            pk[i] = pack_bf16x2(g2.x, g2.y);
          }
          tmem_st16(tDP + hf * 64 + cc * 16, pk);  // dS over this half's own dP columns, already read
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->e_second);
    }
    if (!ok) fail(SITE_BW_ELEM);
    // ---- epilogue: dQ = scale * (dS K) -> bf16
    if (ok && nj > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->acc_done, 0, tmo, abort_flag));
      tc_fence_after();
    }
    if (ok) {
      // every lane loads (tcgen05.ld is warp-collective); rows past T store nothing;
      // each column half writes D/2 columns
      __nv_bfloat16* drow = p.dq + row_index * D + hf * (D / 2);
      const float sc = p.scale;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t a[32];
        if (nj > 0) {
          tmem_ld32(tmem + lane_base + C::COL_ACC + hf * (D / 2) + cc * 32, a);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = 0u;
        }
        if (row_valid) {
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(a[8 * qd + 0]) * sc, __uint_as_float(a[8 * qd + 1]) * sc);
            w.y = pack_bf16x2(__uint_as_float(a[8 * qd + 2]) * sc, __uint_as_float(a[8 * qd + 3]) * sc);
            w.z = pack_bf16x2(__uint_as_float(a[8 * qd + 4]) * sc, __uint_as_float(a[8 * qd + 5]) * sc);
            w.w = pack_bf16x2(__uint_as_float(a[8 * qd + 6]) * sc, __uint_as_float(a[8 * qd + 7]) * sc);
            *reinterpret_cast<uint4*>(drow + cc * 32 + 8 * qd) = w;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// dK, dV: one 128-key tile kt of (batch, KV head) bkv per CTA, looping over the
// stacked query tiles
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void bwd_dkdv_cta(const CUtensorMap& tmQ, const CUtensorMap& tmDO,
                                             const CUtensorMap& tmK, const CUtensorMap& tmV,
                                             const CUtensorMap& tmVec, const BwParams& p, const int kt,
                                             const int bkv) {
  using C = BwCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  uint8_t* sK = smem + C::OFF_FIX;
  uint8_t* sV = sK + C::TILE_BYTES;
  uint8_t* sRing = smem + C::OFF_RING;  // four tile slots (slot_late / slot_early) for Q and dO
  BwBars* bars = reinterpret_cast<BwBars*>(smem + C::OFF_BAR);
  float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC);  // per ring stage: [-lse2 | -D][128]
  uint8_t* sPT = smem + C::OFF_PT;  // P^T of the current step, the A operand of dV
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = bkv / p.Hkv;
  const int kvh = bkv % p.Hkv;
  const int shift = p.S - p.T;
  const int key0 = kt * C::BN;
  // query tiles that see any key of this tile: position pos sees key0 iff key0 <= pos + shift
  int qt0 = 0;
  if (p.causal) qt0 = max(0, key0 - shift) / p.rows_per_head;
  const int nsteps = max(0, p.n_qtiles - qt0);

  if (threadIdx.x == 0) {
    mbar_init(&bars->fix_full, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->e_first, C::EW_THREADS);
    mbar_init(&bars->e_first_odd, C::EW_THREADS);
    mbar_init(&bars->s_read, C::EW_THREADS);
    mbar_init(&bars->pt_free, 1);
    mbar_init(&bars->e_second, C::EW_THREADS);
    mbar_init(&bars->acc_done, 1);
    for (int t = 0; t < 4; ++t) {
      mbar_init(&bars->slot_full[t], 1);
      mbar_init(&bars->slot_empty[t], 1);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::MMA_WARP) tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;
  const uint64_t tmo = p.timeout_ns;
  const uint64_t tmo_unwind = unwind_timeout(tmo);  // copies landing, MMAs draining
  auto fail = [&](unsigned site) {
    record_error(p.err, FA_ERR_TIMEOUT, site);
    *abort_flag = 1;
  };

  if (warp == C::PRODUCER_WARP) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars->fix_full, 2 * C::TILE_BYTES);
      for (int c = 0; c < C::KCH; ++c) {
        tma_load_3d(sK + c * C::CHUNK_BYTES, &tmK, &bars->fix_full, c * 64, key0, bkv);
        tma_load_3d(sV + c * C::CHUNK_BYTES, &tmV, &bars->fix_full, c * 64, key0, bkv);
      }
      int issued = 0;   // steps whose Q and dO loads were both issued
      int q_only = -1;  // a step whose Q load was issued alone
      for (int i = 0; i < nsteps; ++i) {
        // each slot's previous use was step i - 2
        const int qs = slot_late(i), ds = slot_early(i);
        const uint32_t prev = ((i >> 1) - 1) & 1;
        const int qt = qt0 + i;
        if (i >= 2 && !mbar_wait(&bars->slot_empty[qs], prev, tmo, abort_flag)) {
          fail(SITE_BW_PRODUCER);
          break;
        }
        mbar_arrive_expect_tx(&bars->slot_full[qs], C::TILE_BYTES);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(sRing + qs * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmQ, &bars->slot_full[qs], c * 64,
                      qt * p.rows_per_head, kvh * p.g, b);
        q_only = i;
        if (i >= 2 && !mbar_wait(&bars->slot_empty[ds], prev, tmo, abort_flag)) {
          fail(SITE_BW_PRODUCER);
          break;
        }
        if (i == 0) asm volatile("griddepcontrol.wait;" ::: "memory");  // the row pass's values are visible
        // dO, and the tile's -lse2 (plane B + b) and -D (plane b) in stacked row order
        // (positions past T read as 0; their Q and dO rows are zero as well). The
        // vectors' buffer i & 1 was last read by the warps in step i - 2, before dK(i - 2)
        // and so before this slot came back.
        mbar_arrive_expect_tx(&bars->slot_full[ds], C::TILE_BYTES + 2 * C::BM * 4);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(sRing + ds * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmDO, &bars->slot_full[ds], c * 64,
                      qt * p.rows_per_head, kvh * p.g, b);
        tma_load_3d(vec + (i & 1) * 2 * C::BM, &tmVec, &bars->slot_full[ds], qt * p.rows_per_head, kvh * p.g,
                    p.B + b);
        tma_load_3d(vec + (i & 1) * 2 * C::BM + C::BM, &tmVec, &bars->slot_full[ds], qt * p.rows_per_head,
                    kvh * p.g, b);
        q_only = -1;
        issued = i + 1;
      }
      if (*abort_flag) {
        mbar_wait(&bars->fix_full, 0, tmo_unwind);
        for (int x = max(0, issued - 2); x < issued; ++x) {
          mbar_wait(&bars->slot_full[slot_late(x)], (x >> 1) & 1, tmo_unwind);
          mbar_wait(&bars->slot_full[slot_early(x)], (x >> 1) & 1, tmo_unwind);
        }
        if (q_only >= 0) mbar_wait(&bars->slot_full[slot_late(q_only)], (q_only >> 1) & 1, tmo_unwind);
      }
    }
  } else if (warp == C::MMA_WARP) {
    const bool leader = elect_one();
    constexpr uint32_t idesc_ss = idesc_bf16_f32(128, C::BN, 0, 0);
    constexpr uint32_t idesc_ts = idesc_bf16_f32(128, D, 0, 1);
    const uint64_t dKd = smem_desc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t dVd = smem_desc_sw128(smem_u32(sV), 16, 1024);
    const uint64_t dRing = smem_desc_sw128(smem_u32(sRing), 16, 1024);               // Q (for S^T), dO (for dP^T)
    const uint64_t dRingMn = smem_desc_sw128(smem_u32(sRing), C::CHUNK_BYTES, 1024);  // Q (for dK), dO (for dV)
    auto slot_off = [](int t) { return static_cast<uint64_t>((t * C::TILE_BYTES) >> 4); };
    const uint64_t dPT = smem_desc_sw128(smem_u32(sPT), 16, 1024);  // P^T (keys x queries) as the A of dV
    // Issue order: S^T(0), dP^T(0), then per query tile n: S^T(n+1) as soon as the warps
    // have read S^T(n) out of TMEM, dV(n) += P^T(n) dO_n (P^T from shared memory),
    // dK(n) += dS^T(n) Q_n (dS^T over dP^T's columns), dP^T(n+1). So S^T(n+1) runs under
    // the warps' P phase of tile n, and dP^T(n+1) under their P phase of tile n+1. dV(n)
    // gives dO_n's slot and the P^T buffer back, dK(n) Q_n's slot.
    auto issue_s = [&](int n) {
      const uint64_t so = slot_off(slot_late(n));
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4);
          tc_mma_ss(tmem + C::COL_S, dKd + off, dRing + so + off, idesc_ss, kk > 0 ? 1u : 0u);
        }
        tc_commit(&bars->s_full);
      }
    };
    auto issue_dp = [&](int n) {
      const uint64_t so = slot_off(slot_early(n));
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4);
          tc_mma_ss(tmem + C::COL_DP, dVd + off, dRing + so + off, idesc_ss, kk > 0 ? 1u : 0u);
        }
        tc_commit(&bars->dp_full);
      }
    };
    bool ok = mbar_wait(&bars->fix_full, 0, tmo, abort_flag);
    if (ok && nsteps > 0) {
      ok = mbar_wait(&bars->slot_full[slot_late(0)], 0, tmo, abort_flag) &&
           mbar_wait(&bars->slot_full[slot_early(0)], 0, tmo, abort_flag);
      tc_fence_after();
      if (ok) {
        issue_s(0);
        issue_dp(0);
      }
    }
    for (int i = 0; ok && i < nsteps; ++i) {
      const uint32_t use_next = ((i + 1) >> 1) & 1;  // slot parity of step i + 1
      if (i + 1 < nsteps) {
        if (!mbar_wait(&bars->s_read, i & 1, tmo, abort_flag) ||
            !mbar_wait(&bars->slot_full[slot_late(i + 1)], use_next, tmo, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(i + 1);
      }
      if (!mbar_wait((i & 1) ? &bars->e_first_odd : &bars->e_first, (i >> 1) & 1, tmo, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (leader) {
        const int ds = slot_early(i);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4);
          tc_mma_ss(tmem + C::COL_ACC, dPT + off, dRingMn + slot_off(ds) + static_cast<uint64_t>((kk * 2048) >> 4),
                    idesc_ts, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&bars->slot_empty[ds]);
        tc_commit(&bars->pt_free);
      }
      if (!mbar_wait(&bars->e_second, i & 1, tmo, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (leader) {
        const int qs = slot_late(i);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          tc_mma_ts(tmem + C::COL_ACC + D, tmem + C::COL_DP + C::packed_col(kk),
                    dRingMn + slot_off(qs) + static_cast<uint64_t>((kk * 2048) >> 4), idesc_ts,
                    (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&bars->slot_empty[qs]);
      }
      if (i + 1 < nsteps) {
        if (!mbar_wait(&bars->slot_full[slot_early(i + 1)], use_next, tmo, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_dp(i + 1);
      }
    }
    if (!ok && leader) fail(SITE_BW_MMA);
    if (leader) tc_commit(&bars->acc_done);
    mbar_wait(&bars->acc_done, 0, tmo_unwind);
  } else {
    // ---- elementwise warps: one key row per thread pair (TMEM lane), column half
    //      hf; a step's 128 columns are the stacked query rows of one query tile
    const int r = threadIdx.x & 127;
    const int hf = warp >> 2;
    const int key = key0 + r;
    const bool key_valid = key < p.S;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::COL_S;
    const uint32_t tDP = tmem + lane_base + C::COL_DP;
    const float2 c2 = make_float2(p.c, p.c);
    const int rmask = p.rows_per_head - 1;
    bool ok = true;
    for (int i = 0; i < nsteps; ++i) {
      const int qt = qt0 + i;
      // this step's -lse2 and -D of the 128 query columns came with its dO tile
      const float* nl2v = vec + (i & 1) * 2 * C::BM + hf * 64;  // this half's 64 columns
      const float* ndv = nl2v + C::BM;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->slot_full[slot_early(i)], (i >> 1) & 1, tmo, abort_flag) &&
                                       mbar_wait(&bars->s_full, i & 1, tmo, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // column col is position qt * rows_per_head + (col & rmask) of head col / rows_per_head
      // (rows_per_head = 128 / g is a power of two); the key is visible to it iff
      // key <= position + shift, i.e. (col & rmask) >= vis_from
      const int vis_from = p.causal ? key - shift - qt * p.rows_per_head : INT_MIN;
      const bool masked = !__all_sync(0xffffffffu, key_valid && vis_from <= 0);
      // P phase: P^T = 2^(S^T*c - lse2[col]) for this half's 64 query columns, kept in
      // registers for the dS phase and written in bf16 to the shared-memory P^T tile
      float pv[64];
      {
        uint32_t sr[2][32];
        tmem_ld32(tS + hf * 64, sr[0]);
        tmem_ld32(tS + hf * 64 + 32, sr[1]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bars->s_read);  // S^T(i) is in registers: S^T(i+1) may overwrite it
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 l4 = *reinterpret_cast<const float4*>(nl2v + cc * 32 + 4 * q);
            const int e = cc * 32 + 4 * q;
            const float2 x0 = ffma2(make_float2(__uint_as_float(sr[cc][4 * q]), __uint_as_float(sr[cc][4 * q + 1])),
                                    c2, make_float2(l4.x, l4.y));
            const float2 x1 = ffma2(make_float2(__uint_as_float(sr[cc][4 * q + 2]), __uint_as_float(sr[cc][4 * q + 3])),
                                    c2, make_float2(l4.z, l4.w));
            pv[e] = ex2_approx(x0.x);
            pv[e + 1] = ex2_approx(x0.y);
            pv[e + 2] = ex2_approx(x1.x);
            pv[e + 3] = ex2_approx(x1.y);
          }
        }
      }
      if (masked) {  // keys past S, or (causal) columns the key is not visible to
#pragma unroll
        for (int ii = 0; ii < 64; ++ii)
          if (!(key_valid && ((hf * 64 + ii) & rmask) >= vis_from)) pv[ii] = 0.f;
      }
      // the P^T tile is free once dV(i-1) has read it
      if (i > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->pt_free, (i - 1) & 1, tmo, abort_flag))) {
        ok = false;
        break;
      }
      {
        // row r (this key) of chunk hf: 8 16-byte units of 8 queries, 128-byte swizzle
        uint8_t* prow = sPT + hf * C::CHUNK_BYTES + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(prow + ((u ^ (r & 7)) << 4)) =
              make_uint4(pack_bf16x2(pv[8 * u + 0], pv[8 * u + 1]), pack_bf16x2(pv[8 * u + 2], pv[8 * u + 3]),
                         pack_bf16x2(pv[8 * u + 4], pv[8 * u + 5]), pack_bf16x2(pv[8 * u + 6], pv[8 * u + 7]));
      }
      fence_async_smem();  // the tensor core reads the tile through the async proxy
      mbar_arrive((i & 1) ? &bars->e_first_odd : &bars->e_first);
      // dS phase: dS^T = P^T * (dP^T - D[col]) over this half's own dP^T columns
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->dp_full, i & 1, tmo, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        uint32_t dr[2][32];
        tmem_ld32(tDP + hf * 64, dr[0]);
        tmem_ld32(tDP + hf * 64 + 32, dr[1]);
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pd[16];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 d4 = *reinterpret_cast<const float4*>(ndv + cc * 32 + 4 * q);
            const int e = cc * 32 + 4 * q;
            const float2 t0 = fadd2(make_float2(__uint_as_float(dr[cc][4 * q]), __uint_as_float(dr[cc][4 * q + 1])),
                                    make_float2(d4.x, d4.y));
            const float2 t1 = fadd2(make_float2(__uint_as_float(dr[cc][4 * q + 2]), __uint_as_float(dr[cc][4 * q + 3])),
                                    make_float2(d4.z, d4.w));
            const float2 g0 = fmul2(make_float2(pv[e], pv[e + 1]), t0);
            const float2 g1 = fmul2(make_float2(pv[e + 2], pv[e + 3]), t1);
            pd[2 * q] = pack_bf16x2(g0.x, g0.y);
            pd[2 * q + 1] = pack_bf16x2(g1.x, g1.y);
          }
          tmem_st16(tDP + hf * 64 + cc * 16, pd);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->e_second);
    }
    if (!ok) fail(SITE_BW_ELEM);
    // ---- epilogue: dV, dK = scale * (dS^T Q) -> bf16
    if (ok && nsteps > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->acc_done, 0, tmo, abort_flag));
      tc_fence_after();
    }
    if (ok) {
      const size_t krow = static_cast<size_t>(bkv) * p.S + (key_valid ? key : 0);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* drow = (which ? p.dk : p.dv) + krow * D + hf * (D / 2);
        const float sc = which ? p.scale : 1.f;
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          uint32_t a[32];
          if (nsteps > 0) {
            tmem_ld32(tmem + lane_base + C::COL_ACC + which * D + hf * (D / 2) + cc * 32, a);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) a[ii] = 0u;
          }
          if (key_valid) {
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(a[8 * qd + 0]) * sc, __uint_as_float(a[8 * qd + 1]) * sc);
              w.y = pack_bf16x2(__uint_as_float(a[8 * qd + 2]) * sc, __uint_as_float(a[8 * qd + 3]) * sc);
              w.z = pack_bf16x2(__uint_as_float(a[8 * qd + 4]) * sc, __uint_as_float(a[8 * qd + 5]) * sc);
              w.w = pack_bf16x2(__uint_as_float(a[8 * qd + 6]) * sc, __uint_as_float(a[8 * qd + 7]) * sc);
              *reinterpret_cast<uint4*>(drow + cc * 32 + 8 * qd) = w;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Both passes in one launch: the first n_ktiles * B * Hkv CTAs compute dK/dV (heaviest
// key tiles first under the causal mask), the rest dQ (heaviest query tiles first),
// so the last wave of the first pass fills with work of the second. The two passes
// share no data but the inputs.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(320, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmVec, const BwParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the next launch on the stream (for a training loop, the next backward's row pass)
  // may start as SMs free up; it waits for this grid before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (smem_u32(smem_raw) & 1023u) {  // the swizzled tiles need 1024-byte alignment and the layout has no slack
    if (threadIdx.x == 0) record_error(p.err, FA_ERR_BOUNDS, SITE_BW_SMEM);
    return;
  }
  const int n_kv = p.n_ktiles * p.B * p.Hkv;
  const int x = static_cast<int>(blockIdx.x);
  if (x < n_kv) {
    bwd_dkdv_cta<D>(tmQ, tmDO, tmK, tmV, tmVec, p, x % p.n_ktiles, x / p.n_ktiles);
  } else {
    const int y = x - n_kv;
    bwd_dq_cta<D>(tmQ, tmDO, tmK, tmV, p, p.n_qtiles - 1 - y % p.n_qtiles, y / p.n_qtiles);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();

static bool encode_stacked(EncodeTiledFn enc, CUtensorMap* m, const void* base, int B, int Hq, int T, int d, int g,
                           int rows_per_head) {
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)Hq, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)T * d * 2, (cuuint64_t)Hq * T * d * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)rows_per_head, (cuuint32_t)g, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool encode_keys(EncodeTiledFn enc, CUtensorMap* m, const void* base, int B, int Hkv, int S, int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)B * Hkv};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)S * d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static int launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tvec, const BwParams& p, cudaStream_t stream) {
  using C = BwCfg<D>;
  auto kfn = bwd_kernel<D>;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  const unsigned nbkv = static_cast<unsigned>(p.B * p.Hkv);
  const long long ctas = static_cast<long long>(p.n_ktiles + p.n_qtiles) * nbkv;
  if (ctas > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  // a programmatic dependent of the row pass: its CTAs start (barriers, TMEM, the fixed
  // tiles, the first products) while the row pass finishes, and wait only where they
  // read its values
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kfn, tq, tdo, tk, tv, tvec, p) != cudaSuccess) return FA_ERR_CUDA;
  return launch_status();
}

// q, o, d_o [B][Hq][T][d]; k, v [B][Hkv][S][d] bf16; lse [B][Hq][T] fp32; vecs:
// 2 * B*Hq*T_pad floats of scratch for the row vectors (T_pad = T rounded up to 4).
// Writes dq, dk, dv (bf16, shapes of q, k, v).
int launch_backward(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* d_o,
                    void* dq, void* dk, void* dv, float* vecs, int B, int Hq, int Hkv, int T, int S, int d,
                    float scale, int causal, cudaStream_t stream, unsigned* err, unsigned long long timeout_ns) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return FA_ERR_CUDA;
  const int g = Hq / Hkv;
  const int rows_per_head = 128 / g;
  CUtensorMap tq, tdo, tk, tv;
  if (!encode_stacked(enc, &tq, q, B, Hq, T, d, g, rows_per_head) ||
      !encode_stacked(enc, &tdo, d_o, B, Hq, T, d, g, rows_per_head) || !encode_keys(enc, &tk, k, B, Hkv, S, d) ||
      !encode_keys(enc, &tv, v, B, Hkv, S, d))
    return FA_ERR_CUDA;
  const int T_pad = (T + 3) / 4 * 4;
  CUtensorMap tvec;
  {
    // planes: -D of batch b at b, -lse2 of batch b at B + b; rows T_pad floats apart
    cuuint64_t dims[3] = {(cuuint64_t)T, (cuuint64_t)Hq, (cuuint64_t)2 * B};
    cuuint64_t strides[2] = {(cuuint64_t)T_pad * 4, (cuuint64_t)Hq * T_pad * 4};
    cuuint32_t box[3] = {(cuuint32_t)rows_per_head, (cuuint32_t)g, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tvec, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, vecs, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FA_ERR_CUDA;
  }
  const long long rows = static_cast<long long>(B) * Hq * T;
  const long long rows_per_block = 256 / (d / 16);
  {
    // a programmatic dependent of the launch before it on the stream (it waits before
    // reading anything)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + rows_per_block - 1) / rows_per_block));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, bwd_rowsum_kernel, static_cast<const __nv_bfloat16*>(o),
                           static_cast<const __nv_bfloat16*>(d_o), lse, vecs, rows, T, T_pad, d) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  BwParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.neg_d = vecs;
  p.nl2 = vecs + static_cast<size_t>(B) * Hq * T_pad;
  p.T_pad = T_pad;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.T = T;
  p.S = S;
  p.g = g;
  p.rows_per_head = rows_per_head;
  p.n_qtiles = (T + rows_per_head - 1) / rows_per_head;
  p.n_ktiles = (S + 127) / 128;
  p.causal = causal;
  p.scale = scale;
  p.c = scale * kLog2e;
  p.err = err;
  p.timeout_ns = timeout_ns;
  return d == 128 ? launch_bwd_t<128>(tq, tdo, tk, tv, tvec, p, stream)
                  : launch_bwd_t<64>(tq, tdo, tk, tv, tvec, p, stream);
}

}  // namespace fa
