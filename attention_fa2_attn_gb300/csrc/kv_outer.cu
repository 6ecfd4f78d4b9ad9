// kv_outer.cu -- attention forward in the FlashAttention-1 loop order on the
// sm_103a tensor cores, the measured contrast to the FlashAttention-2 order of
// prefill_tc.cu.
//
// What it computes ("Kernel visualization: Flash Attention 1", "The tiled
// version", "Kernel implementation" and "Counting trips across HBM"): the
// key/value tiles are the outer loop and the query tiles the inner one. For each
// (K_j, V_j), every query tile i brings its Q_i and its running state from HBM --
// the max m, the sum l and the output O', kept normalised -- folds the key tile
// in and writes m, l and O' back:
//   x     = scale * Q_i K_j^T                   (masked scores are -inf)
//   m_new = max(m, rowmax(x))
//   l_new = l e^(m - m_new) + rowsum(e^(x - m_new))
//   O'    = (l e^(m - m_new) O' + e^(x - m_new) V_j) / l_new
// After a tile's last key tile O' is the attention output. Q, O', m and l cross
// HBM once per key tile, where the FlashAttention-2 order reads Q and writes O
// once. (The exponentials run in base 2 on x * log2(e); the values are the same.)
//
// How (GB300-specific):
//   * one CTA per (batch, query head), the pages' grid, or per (batch, query
//     head, band of query tiles) when row_bands > 1 so the grid can fill the
//     SMs; a CTA runs the loop nest over its band and loads K_j, V_j once per band.
//   * the running state is a caller-provided fp32 workspace: O' [B][Hq][T][d] and
//     m, l [B][Hq][T]. O' tiles travel by TMA (128-byte-swizzled boxes of 32 fp32
//     columns) into two shared-memory buffers and back out; m and l are plain
//     per-row loads and stores (thread r owns row r of the tile).
//   * warp 5 (one elected lane) issues S = Q_i K_j^T (both operands in smem) and
//     PV = P V_j (P from TMEM, where the softmax left it) into TMEM, alternating
//     between two column sets on consecutive steps. Warp 4 (one lane) is the TMA
//     producer: K_j and V_j, Q_i, the O' tile in, and the finished O' tile out.
//     Warps 0-3 run the softmax of step s, then the O' update of step s-1, so the
//     PV product of a step runs under the softmax of the next.
//   * a tile's first key tile starts from m = -inf, l = 0, O' = 0 without reading
//     the workspace; its last one writes bf16 O and lse instead of O', m and l.
//   * causal (bottom-right): a tile is visited only for key tiles that hold a key
//     visible to one of its rows; the mask is applied per element.
// Every mbarrier wait is bounded (%globaltimer); a wait that runs out records
// FA_ERR_TIMEOUT in the device error word and the CTA unwinds, frees TMEM and
// returns.
#include "common.cuh"

namespace fa {

template <int D>
struct KoCfg {
  static constexpr int BM = 128;                 // query rows per tile (TMEM lanes)
  static constexpr int BN = 128;                 // keys per K/V tile
  static constexpr int KCH = D / 64;             // bf16 128-byte chunks along d
  static constexpr int OCH = D / 32;             // fp32 128-byte boxes along d
  static constexpr int CHUNK_BYTES = 128 * 128;  // one 128-row x 128-byte swizzled chunk
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int O_BYTES = BM * D * 4;     // one fp32 O' tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_Q = OFF_V + KV_BYTES;
  static constexpr int OFF_O = OFF_Q + Q_BYTES;  // two O' buffers
  static constexpr int OFF_BAR = OFF_O + 2 * O_BYTES;
  static constexpr int SMEM_USED = OFF_BAR + 256 + 1024;  // + slack to align the base to 1024
  // every CTA allocates all 512 TMEM columns, so no two may share an SM: at
  // d = 64 the request is raised past half of the SM's shared memory
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static constexpr int THREADS = 192;
  static constexpr int PRODUCER_WARP = 4;
  static constexpr int MMA_WARP = 5;
  static constexpr int TMEM_COLS = 512;  // per step parity: 128 S/P columns, then 128 PV columns
};
static_assert(KoCfg<128>::SMEM <= 232448, "shared memory of the d = 128 kernel");

struct KoBars {
  uint64_t kv_full, kv_empty;  // K_j and V_j landed / every MMA reading them completed
  uint64_t q_full, q_empty;    // Q_i landed / S read it
  uint64_t s_full[2];          // per step parity: S in TMEM
  uint64_t p_full[2];          // P written over S (128 arrivals)
  uint64_t pv_full[2];         // PV in TMEM
  uint64_t o_full[2];          // per O' buffer: the tile's O' landed (or nothing to load)
  uint64_t o_ready[2];         // per O' buffer: the update warps are done with it (128 arrivals)
  uint64_t drain;              // every MMA the CTA issued has completed (before TMEM is freed)
  uint32_t tmem_base;
  int abort_flag;
};

struct KoParams {
  __nv_bfloat16* o;
  float* lse;
  float* m_ws;  // running max (log2 units) [B*Hq*T]
  float* l_ws;  // running sum [B*Hq*T]
  int B, Hq, Hkv, T, S;
  int g;          // query heads per KV head
  int causal;
  int row_bands;  // CTAs per (batch, query head)
  int n_qt, n_kt;
  float c;  // scale * log2(e)
  unsigned* err;
  unsigned long long timeout_ns;
};

// Last key tile that query tile i needs; -1 when none of its rows sees a key.
__device__ __forceinline__ int ko_jmax(const KoParams& p, int i) {
  if (!p.causal) return p.n_kt - 1;
  const int last_key = min(p.T, (i + 1) * 128) - 1 + (p.S - p.T);  // bottom-right: row r sees keys <= r + S - T
  return last_key < 0 ? -1 : min(p.n_kt - 1, last_key / 128);
}

// The loop nest of one CTA: key tiles j outer, the band's query tiles i in
// [i0, i1) inner, skipping tiles that need no key of tile j (ko_jmax grows with
// i, so those are a prefix of the band).
struct KoIter {
  int i, j, i0, i1;
  __device__ __forceinline__ bool start(const KoParams& p, int lo, int hi) {
    i0 = lo;
    i1 = hi;
    j = 0;
    i = i0;
    while (i < i1 && ko_jmax(p, i) < j) ++i;
    return i < i1;
  }
  __device__ __forceinline__ bool next(const KoParams& p) {
    if (++i < i1) return true;
    ++j;
    i = i0;
    while (i < i1 && ko_jmax(p, i) < j) ++i;
    return i < i1;
  }
};

template <int D>
__global__ void __launch_bounds__(KoCfg<D>::THREADS, 1)
    kv_outer_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const KoParams p) {
  using C = KoCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sO = smem + C::OFF_O;
  KoBars* bars = reinterpret_cast<KoBars*>(smem + C::OFF_BAR);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x / p.row_bands;  // b * Hq + h
  const int band = blockIdx.x % p.row_bands;
  const int b = bh / p.Hq;
  const int kv_plane = b * p.Hkv + (bh % p.Hq) / p.g;
  const int i_lo = static_cast<int>(static_cast<long long>(band) * p.n_qt / p.row_bands);
  const int i_hi = static_cast<int>(static_cast<long long>(band + 1) * p.n_qt / p.row_bands);

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->p_full[x], 128);
      mbar_init(&bars->pv_full[x], 1);
      mbar_init(&bars->o_full[x], 1);
      mbar_init(&bars->o_ready[x], 128);
    }
    mbar_init(&bars->drain, 1);
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
    // ======================= TMA producer (one lane) =======================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmO);
      // steps s-2 and s-1: query tile and whether it was the tile's last key tile
      // (its O' then went to HBM as bf16 O directly and is not stored from smem)
      int e_i[2] = {0, 0};
      bool e_last[2] = {false, false};
      int retired = 0;  // steps whose O' buffer has been handed back, in order
      bool ok = true;
      // wait until the update warps are done with step t's O' buffer and, unless
      // that was the tile's last key tile, store it
      auto retire = [&](int t) -> bool {
        const int ob = t & 1;
        if (!mbar_wait(&bars->o_ready[ob], (t >> 1) & 1, tmo, abort_flag)) return false;
        const int ti = ob ? e_i[1] : e_i[0];
        const bool tl = ob ? e_last[1] : e_last[0];
        if (!tl) {
          for (int c = 0; c < C::OCH; ++c)
            tma_store_3d(&tmO, sO + ob * C::O_BYTES + c * C::CHUNK_BYTES, c * 32, ti * 128, bh);
          bulk_commit_group();
        }
        return true;
      };
      KoIter s_it;
      int s = 0, jidx = -1, prev_j = -1;
      // loads issued so far on kv_full, q_full and the o_full pair (steps armed):
      // each barrier's earlier phases completed before its next load was issued
      int kv_loads = 0, q_loads = 0, o_steps = 0;
      for (bool more = s_it.start(p, i_lo, i_hi); more && !*abort_flag; more = s_it.next(p), ++s) {
        const int i = s_it.i, j = s_it.j;
        const bool new_j = j != prev_j;
        if (new_j) {
          ++jidx;
          if (jidx > 0 && !mbar_wait(&bars->kv_empty, (jidx - 1) & 1, tmo, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->kv_full, 2 * C::KV_BYTES);
          for (int c = 0; c < C::KCH; ++c) {
            tma_load_3d(sK + c * C::CHUNK_BYTES, &tmK, &bars->kv_full, c * 64, j * 128, kv_plane);
            tma_load_3d(sV + c * C::CHUNK_BYTES, &tmV, &bars->kv_full, c * 64, j * 128, kv_plane);
          }
          ++kv_loads;
        }
        if (s > 0 && !mbar_wait(&bars->q_empty, (s - 1) & 1, tmo, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars->q_full, C::Q_BYTES);
        for (int c = 0; c < C::KCH; ++c) tma_load_3d(sQ + c * C::CHUNK_BYTES, &tmQ, &bars->q_full, c * 64, i * 128, bh);
        ++q_loads;
        // this step's O' buffer last held step s-2's tile
        if (s >= 2 && retired <= s - 2) {
          if (!retire(s - 2)) {
            ok = false;
            break;
          }
          retired = s - 1;
          bulk_wait_read_all();
        }
        // a new key tile reads O' tiles the previous key tile wrote: every store
        // of the previous key tile completes first
        if (new_j && s >= 1) {
          if (retired <= s - 1) {
            if (!retire(s - 1)) {
              ok = false;
              break;
            }
            retired = s;
          }
          bulk_wait_all();
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        const bool last = j == ko_jmax(p, i);
        if (s & 1) {
          e_i[1] = i;
          e_last[1] = last;
        } else {
          e_i[0] = i;
          e_last[0] = last;
        }
        uint64_t* of = &bars->o_full[s & 1];
        if (j == 0) {
          mbar_arrive(of);  // first key tile: the state starts empty, nothing to load
        } else {
          mbar_arrive_expect_tx(of, C::O_BYTES);
          for (int c = 0; c < C::OCH; ++c)
            tma_load_3d(sO + (s & 1) * C::O_BYTES + c * C::CHUNK_BYTES, &tmO, of, c * 32, i * 128, bh);
        }
        o_steps = s + 1;
        prev_j = j;
      }
      // hand back (and store) the last steps' buffers
      for (int t = retired; ok && t < s && !*abort_flag; ++t)
        if (!retire(t)) ok = false;
      bulk_wait_all();
      if (!ok) fail(SITE_KO_PRODUCER);
      if (*abort_flag) {
        // loads still in flight must land before the CTA exits: at most the last
        // phase of kv_full and q_full, and the last step of each O' buffer
        if (kv_loads > 0) mbar_wait(&bars->kv_full, (kv_loads - 1) & 1, tmo_unwind);
        if (q_loads > 0) mbar_wait(&bars->q_full, (q_loads - 1) & 1, tmo_unwind);
        for (int t = max(0, o_steps - 2); t < o_steps; ++t) mbar_wait(&bars->o_full[t & 1], (t >> 1) & 1, tmo_unwind);
      }
    }
  } else if (warp == C::MMA_WARP) {
    // ======================= MMA issuer =======================
    const bool leader = elect_one();
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, C::BN, 0, 0);  // A = Q (K-major), B = K (K-major)
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);      // A = P (TMEM), B = V (MN-major)
    const uint64_t dQ = smem_desc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dK = smem_desc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t dV = smem_desc_sw128(smem_u32(sV), C::CHUNK_BYTES, 1024);
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool { return mbar_wait(bar, parity, tmo, abort_flag); };
    // PV of step t into its column set: P (16 keys = 8 columns per MMA) from TMEM
    auto issue_pv = [&](int t) -> bool {
      const int tb = t & 1;
      if (!wwait(&bars->p_full[tb], (t >> 1) & 1)) return false;
      tc_fence_after();
      const uint32_t aP = tmem + tb * 256;
      const uint32_t dO = tmem + tb * 256 + 128;
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          tc_mma_ts(dO, aP + kk * 8, dV + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv, kk > 0 ? 1u : 0u);
        tc_commit(&bars->pv_full[tb]);
      }
      __syncwarp();
      return true;
    };
    bool ok = true;
    KoIter s_it;
    int s = 0, jidx = -1, prev_j = -1;
    bool pv_prev_done = true;  // PV of step s-1 issued
    for (bool more = s_it.start(p, i_lo, i_hi); more && !*abort_flag; more = s_it.next(p), ++s) {
      const int tb = s & 1;
      if (s_it.j != prev_j) {
        // the previous key tile's last PV goes first: K/V are reloaded after it
        if (!pv_prev_done) {
          if (!issue_pv(s - 1)) {
            ok = false;
            break;
          }
          pv_prev_done = true;
        }
        if (s > 0 && leader) tc_commit(&bars->kv_empty);
        __syncwarp();
        ++jidx;
        if (!wwait(&bars->kv_full, jidx & 1)) {
          ok = false;
          break;
        }
      }
      if (!wwait(&bars->q_full, s & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (leader) {
        const uint32_t dS = tmem + tb * 256;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4);
          tc_mma_ss(dS, dQ + off, dK + off, idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(&bars->s_full[tb]);
        tc_commit(&bars->q_empty);
      }
      __syncwarp();
      if (!pv_prev_done) {
        if (!issue_pv(s - 1)) {
          ok = false;
          break;
        }
      }
      pv_prev_done = false;
      prev_j = s_it.j;
    }
    if (ok && !pv_prev_done && !*abort_flag && !issue_pv(s - 1)) ok = false;
    if (!ok) fail(SITE_KO_MMA);
    // every MMA issued must finish before TMEM is released
    if (leader) tc_commit(&bars->drain);
    __syncwarp();
    mbar_wait(&bars->drain, 0, tmo_unwind);
  } else {
    // ============ softmax and O' update: warps 0-3, thread r = row r ============
    const int r = threadIdx.x;  // 0..127
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int shift = p.S - p.T;
    const float c = p.c;
    const float2 c2 = make_float2(c, c);
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool { return mbar_wait(bar, parity, tmo, abort_flag); };
    // query tiles of the band that no key reaches: O = 0, lse = -inf
    for (int i = i_lo; i < i_hi; ++i) {
      if (ko_jmax(p, i) >= 0) break;  // ko_jmax grows with i
      const int row = i * 128 + r;
      if (row >= p.T) break;
      const size_t ridx = static_cast<size_t>(bh) * p.T + row;
      uint4* orow = reinterpret_cast<uint4*>(p.o + ridx * D);
      for (int q = 0; q < D / 8; ++q) orow[q] = make_uint4(0u, 0u, 0u, 0u);
      if (p.lse) p.lse[ridx] = -INFINITY;
    }
    // what the update of a step needs from its softmax
    struct Pend {
      int t, i;
      bool first, last;
      float ca, cb, lse;
    };
    bool ok = true;
    // O' update of step u.t: O' = ca O'_old + cb PV, back into the buffer for the
    // producer to store, or (last key tile) bf16 O and lse to HBM
    auto update = [&](const Pend& u) -> bool {
      const int tb = u.t & 1;
      if (!wwait(&bars->pv_full[tb], (u.t >> 1) & 1)) return false;
      if (!wwait(&bars->o_full[tb], (u.t >> 1) & 1)) return false;
      tc_fence_after();
      const int row = u.i * 128 + r;
      const bool valid = row < p.T;
      const size_t ridx = static_cast<size_t>(bh) * p.T + row;
      uint8_t* obuf = sO + tb * C::O_BYTES + r * 128;
#pragma unroll
      for (int cc = 0; cc < C::OCH; ++cc) {
        uint32_t pv[32];
        tmem_ld32(tmem + lane_base + tb * 256 + 128 + cc * 32, pv);
        tmem_ld_wait();
        float o[32];
        if (u.first) {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0.f;
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(obuf + cc * C::CHUNK_BYTES + ((q ^ (r & 7)) << 4));
            o[4 * q + 0] = v.x;
            o[4 * q + 1] = v.y;
            o[4 * q + 2] = v.z;
            o[4 * q + 3] = v.w;
          }
        }
        const float2 ca2 = make_float2(u.ca, u.ca);
        const float2 cb2 = make_float2(u.cb, u.cb);
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const float2 x = ffma2(make_float2(o[k], o[k + 1]), ca2,
                                 fmul2(make_float2(__uint_as_float(pv[k]), __uint_as_float(pv[k + 1])), cb2));
          o[k] = x.x;
          o[k + 1] = x.y;
        }
        if (u.last) {
          if (valid) {
            uint4* orow = reinterpret_cast<uint4*>(p.o + ridx * D + cc * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              orow[q] = make_uint4(pack_bf16x2(o[8 * q + 0], o[8 * q + 1]), pack_bf16x2(o[8 * q + 2], o[8 * q + 3]),
                                   pack_bf16x2(o[8 * q + 4], o[8 * q + 5]), pack_bf16x2(o[8 * q + 6], o[8 * q + 7]));
          }
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(obuf + cc * C::CHUNK_BYTES + ((q ^ (r & 7)) << 4)) =
                make_float4(o[4 * q + 0], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
      }
      if (u.last && valid && p.lse) p.lse[ridx] = u.lse;
      // PV read out (the next PV into these columns is issued only after this
      // thread's arrival on p_full two steps later); smem writes made visible to
      // the TMA store
      tc_fence_before();
      fence_async_smem();
      mbar_arrive(&bars->o_ready[tb]);
      return true;
    };

    Pend prev{0, 0, false, false, 0.f, 0.f, 0.f};
    bool have_prev = false;
    KoIter s_it;
    int s = 0;
    for (bool more = s_it.start(p, i_lo, i_hi); more && !*abort_flag; more = s_it.next(p), ++s) {
      const int i = s_it.i, j = s_it.j;
      const int tb = s & 1;
      const bool first = j == 0;
      const bool last = j == ko_jmax(p, i);
      const int row = i * 128 + r;
      const bool valid = row < p.T;
      const size_t ridx = static_cast<size_t>(bh) * p.T + row;
      float m_old = -INFINITY, l_old = 0.f;
      if (!first && valid) {
        m_old = p.m_ws[ridx];
        l_old = p.l_ws[ridx];
      }
      if (!wwait(&bars->s_full[tb], (s >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tmem + lane_base + tb * 256;
      uint32_t raw[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, raw[cc]);
      tmem_ld_wait();
      float sc[128];
#pragma unroll
      for (int k = 0; k < 128; ++k) sc[k] = __uint_as_float(raw[k >> 5][k & 31]);
      const int key0 = j * C::BN;
      // keys key0 + k with k > lim are masked: past S, or (causal) past row + S - T
      const int lim = (p.causal ? min(p.S - 1, row + shift) : p.S - 1) - key0;
      if (lim < C::BN - 1) {
#pragma unroll
        for (int k = 0; k < 128; ++k)
          if (k > lim) sc[k] = -INFINITY;
      }
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float a = fmax3(sc[16 * k], sc[16 * k + 1], sc[16 * k + 2]);
#pragma unroll
        for (int x = 3; x < 15; x += 2) a = fmax3(a, sc[16 * k + x], sc[16 * k + x + 1]);
        mx8[k] = fmaxf(a, sc[16 * k + 15]);
      }
      const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
      const float m_new = fmaxf(m_old, mx * c);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // nothing visible yet: every p is 0
      const float2 nm2 = make_float2(-m_use, -m_use);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int e = cc * 32 + 2 * x;
          const float2 y = ffma2(make_float2(sc[e], sc[e + 1]), c2, nm2);
          const float2 ev = make_float2(ex2_approx(y.x), ex2_approx(y.y));
          acc[x & 3] = fadd2(acc[x & 3], ev);
          pk[x] = pack_bf16x2(ev.x, ev.y);
        }
        tmem_st16(tS + cc * 16, pk);  // keys 32cc .. 32cc+31 -> columns 16cc .. 16cc+15
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_full[tb]);
      const float2 at = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
      const float alpha = ex2_approx(m_old - m_use);  // 0 while nothing was seen
      const float l_new = fmaf(l_old, alpha, at.x + at.y);
      Pend cur;
      cur.t = s;
      cur.i = i;
      cur.first = first;
      cur.last = last;
      cur.ca = l_new > 0.f ? l_old * alpha / l_new : 0.f;
      cur.cb = l_new > 0.f ? 1.f / l_new : 0.f;
      cur.lse = l_new > 0.f ? (m_new + log2f(l_new)) * kLn2 : -INFINITY;
      if (!last && valid) {
        p.m_ws[ridx] = m_new;
        p.l_ws[ridx] = l_new;
      }
      if (have_prev && !update(prev)) {
        ok = false;
        break;
      }
      prev = cur;
      have_prev = true;
    }
    if (ok && have_prev && !*abort_flag && !update(prev)) ok = false;
    if (!ok) fail(SITE_KO_UPDATE);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();  // defined in api.cu

// Workspace layout (fa_fwd_kv_outer_workspace_bytes): O' fp32 [B*Hq*T][d], padded
// to 256 bytes, then m [B*Hq*T] and l [B*Hq*T], fp32.
int launch_kv_outer(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int T,
                    int S, int d, float scale, int causal, int row_bands, void* workspace, cudaStream_t stream,
                    unsigned* err, unsigned long long timeout_ns) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return FA_ERR_CUDA;
  const size_t rows = static_cast<size_t>(B) * Hq * T;
  float* o_ws = static_cast<float*>(workspace);
  float* m_ws = o_ws + ((rows * d * 4 + 255) / 256) * 64;
  float* l_ws = m_ws + rows;
  CUtensorMap tq, tk, tv, to;
  const cuuint32_t es[3] = {1, 1, 1};
  {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)B * Hq};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)T * d * 2};
    cuuint32_t box[3] = {64, 128, 1};
    if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FA_ERR_CUDA;
  }
  for (int w = 0; w < 2; ++w) {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)B * Hkv};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)S * d * 2};
    cuuint32_t box[3] = {64, 128, 1};
    if (enc(w == 0 ? &tk : &tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w == 0 ? k : v), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FA_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)B * Hq};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)T * d * 4};
    cuuint32_t box[3] = {32, 128, 1};
    if (enc(&to, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, o_ws, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FA_ERR_CUDA;
  }
  KoParams p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.m_ws = m_ws;
  p.l_ws = l_ws;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.T = T;
  p.S = S;
  p.g = Hq / Hkv;
  p.causal = causal;
  p.n_qt = (T + 127) / 128;
  p.n_kt = (S + 127) / 128;
  p.row_bands = row_bands < p.n_qt ? row_bands : p.n_qt;
  p.c = scale * kLog2e;
  p.err = err;
  p.timeout_ns = timeout_ns;
  const long long grid = static_cast<long long>(B) * Hq * p.row_bands;
  if (grid > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (d == 128) {
    auto kfn = kv_outer_kernel<128>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, KoCfg<128>::SMEM) != cudaSuccess)
      return FA_ERR_CUDA;
    kfn<<<static_cast<int>(grid), KoCfg<128>::THREADS, KoCfg<128>::SMEM, stream>>>(tq, tk, tv, to, p);
  } else {
    auto kfn = kv_outer_kernel<64>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, KoCfg<64>::SMEM) != cudaSuccess)
      return FA_ERR_CUDA;
    kfn<<<static_cast<int>(grid), KoCfg<64>::THREADS, KoCfg<64>::SMEM, stream>>>(tq, tk, tv, to, p);
  }
  return launch_status();
}

}  // namespace fa
