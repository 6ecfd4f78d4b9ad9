// prefill_tc.cu -- fused attention forward on the sm_103a tensor cores.
//
// What it computes (per query row, "Kernel visualization: Flash Attention 1",
// "The tiled version"; "Softmax and FlashAttention", "Concept" and "Maths"):
// stream the keys in tiles of BN, keep the running max m, running sum l and
// the unnormalised output u of every row, rescale l and u by 2^(m_old - m_new)
// when the max rises, and divide by l once after the last tile (the
// FlashAttention-2 order of "Attention kernel chains", "The online softmax on
// numbers"). lse = ln2 * (m + log2 l) is written per row ("What the backward
// pass saves").
//
// How (GB300-specific):
//   * one CTA per (batch, KV head, pair of BM = 128-row query tiles). With GQA
//     the g query heads of a group are stacked as rows of a tile (128/g
//     positions x g heads), so every K/V tile is loaded once per group and
//     serves 256 rows ("GQA loads KV once per group"). A 4-D TMA box
//     {64, 128/g, g, 1} over Q [B][Hq][T][d] builds a stacked tile directly.
//   * warp 8 (one elected thread): TMA producer. Both Q tiles once, then K_j
//     and V_j into a 2-stage ring of 128-byte-swizzled shared-memory tiles,
//     with separate full/empty mbarriers for K and V.
//   * warp 9: allocates all 512 TMEM columns -- per query tile t a 128-column
//     S/P region and a d-column O region -- and one thread issues the
//     tcgen05.mma chain. The two query tiles ping-pong on the tensor core:
//     while one tile's softmax runs, the MMAs of the other tile proceed.
//     S_t = Q_t K_j^T reads both operands from smem; O_t += P_t V_j reads P_t
//     from TMEM (where the softmax left it) and V_j from smem (MN-major).
//   * warps 0-3 / 4-7: the softmax of tile 0 / 1, thread r = row r = TMEM
//     lane r. tcgen05.ld of S, row max, p = 2^(s*c - m) with c =
//     scale*log2(e) folded into one packed FFMA, P packed to bf16 and written
//     back over S with tcgen05.st. O is rescaled in TMEM only when the max of
//     some row of the warp rose.
//   * causal: tiles entirely above the diagonal are never loaded or issued;
//     the mask is evaluated only on tiles that cross it (or the ragged end).
//     CTAs are ordered heaviest first.
// Every mbarrier wait is bounded (%globaltimer); a wait that runs out records
// FA_ERR_TIMEOUT in the device error word and the CTA unwinds, frees TMEM and
// returns.
#include "common.cuh"

namespace fa {

template <int D>
struct PfCfg {
  static constexpr int BM = 128;                 // query rows per tile (TMEM lanes)
  static constexpr int QT = 2;                   // query tiles per CTA
  static constexpr int BN = 128;                 // keys per K/V tile
  static constexpr int KCH = D / 64;             // 64-element (128-byte) chunks along d
  static constexpr int STAGES = 2;               // K/V ring depth
  static constexpr int CHUNK_BYTES = 128 * 128;  // one 128-row x 128-byte swizzled chunk
  static constexpr int Q_BYTES = BM * D * 2;     // one query tile
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QT * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_BYTES;
  static constexpr int BAR_BYTES = 256;
  // paged: the batch's sequences ranked by key count (longest first), for the item order
  static constexpr int MAX_RANKED = 512;
  static constexpr int OFF_ORDER = OFF_BAR + BAR_BYTES;
  static constexpr int SMEM = OFF_ORDER + 1024;                     // + slack to align the base to 1024
  static constexpr int SMEM_PAGED = OFF_ORDER + MAX_RANKED * 4 + 1024;
  static constexpr int TMEM_COLS = 512;
  static constexpr int TILE_COLS = 256;   // TMEM columns per query tile: S/P then O
  static constexpr int O_OFF = 128;       // O region inside a tile's columns
  // warpgroups 0 and 1: softmax of tile 0 and 1; warpgroup 2: producer warp,
  // MMA warp and two idle warps. Launched at 168 registers a thread; warpgroup
  // 2 gives back down to 120 and the softmax warpgroups take up to 192:
  // 256 * 192 + 128 * 120 = 64512 = 384 * 168.
  static constexpr int THREADS = 384;
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
  static constexpr int SOFTMAX_REGS = 192;
  static constexpr int AUX_REGS = 120;
};

struct PfParams {
  __nv_bfloat16* o;
  float* lse;
  int B, Hq, Hkv, T, S;
  int g;              // query heads per KV head
  int rows_per_head;  // 128 / g query positions per tile
  int n_qtiles;       // ceil(T / rows_per_head)
  int n_pairs;        // ceil(n_qtiles / 2)
  int n_items;        // n_pairs * B * Hkv work items, taken round-robin by the persistent CTAs
  int causal;
  float c;            // scale * log2(e)
  unsigned* err;
  unsigned long long timeout_ns;
  // paged K/V only: pools [num_pages][16][Hkv][d], block_table [B][max_pages], seqlens [B]
  const int* block_table;
  const int* seqlens;
  int max_pages, num_pages;
  // key split only: num_splits ranges of split_tiles 128-key tiles each; partials
  // o_part [num_splits][B*Hq*T][D] fp32 (normalised) and lse_part [num_splits][B*Hq*T]
  int num_splits, split_tiles;
  float* o_part;
  float* lse_part;
};

struct PfBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[2], v_full[2], k_empty[2], v_empty[2];
  uint64_t s_full[2];   // per query tile: S_t(j) computed
  uint64_t p_full[2];   // per query tile: P_t(j) in TMEM (and O_t rescaled)
  uint64_t pv_done[2];  // per query tile: the item's last O_t += P_t V finished (once per item)
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// One work item: a pair of 128-row query tiles of one (batch, KV head).
struct PfItem {
  int b, kvh, bh;
  int p0[2];  // first query position of tile 0 / 1
  int nj[2];  // key tiles tile 0 / 1 needs (0 for a tile past T)
};

// Keys of sequence b: p.S, or (paged) its seqlens entry clamped to the table's reach.
// Not carried in PfItem: the contiguous kernel keeps that struct as small as possible.
template <bool PAGED>
__device__ __forceinline__ int item_keys(const PfParams& p, int b) {
  return PAGED ? max(0, min(__ldg(p.seqlens + b), p.max_pages * 16)) : p.S;
}

// Key split: item `it` covers key tiles split_j0 .. of range it % num_splits.
template <bool SPLIT>
__device__ __forceinline__ int split_j0(const PfParams& p, int it) {
  return SPLIT ? (it % p.num_splits) * p.split_tiles : 0;
}

// Snake dealing of items sorted heaviest first: slot `it` of CTA x in round
// it / G takes sorted item round * G + x, or round * G + (G - 1 - x) when the
// round runs backwards. The snake is anchored at the end: the last full round
// runs backwards, the one before it forwards, and so on. So the CTAs with the
// lowest indexes end the full rounds the least loaded, and they are the ones
// that take the last, partial round (forwards, as only CTAs 0 .. n % G - 1 get
// a slot in it). A reversed round stays inside its own G items, so the map is
// one to one.
__device__ __forceinline__ int snake_sorted(int it, int n_items) {
  const int G = gridDim.x;
  const int round = it / G;
  const int x = it - round * G;
  const int full_rounds = n_items / G;
  return ((full_rounds - round) & 1) ? round * G + (G - 1 - x) : it;
}

template <bool PAGED, bool SPLIT = false>
__device__ __forceinline__ PfItem pf_item(const PfParams& p, int it, int bn, const int* order) {
  PfItem w;
  const int bh_count = p.B * p.Hkv;
  int qp;
  if (SPLIT) {
    // low-occupancy shapes: (query-tile pair, key range) units, head-major
    const int base = it / p.num_splits;
    w.bh = base / p.n_pairs;
    qp = base % p.n_pairs;
  } else if (PAGED) {
    // Sequences of a paged batch differ in length, so item weights differ by
    // sequence: items go longest sequence first (order[] ranks them when the batch
    // has at most MAX_RANKED sequences), within it heaviest query-tile pair first,
    // dealt to the CTAs in snake order.
    const int sorted = snake_sorted(it, p.n_items);
    const int per_b = p.Hkv * p.n_pairs;
    const int rank = sorted / per_b;
    const int within = sorted - rank * per_b;
    const int b = order ? order[rank] : rank;
    qp = p.n_pairs - 1 - within / p.Hkv;
    w.bh = b * p.Hkv + within % p.Hkv;
  } else if (p.causal) {
    // items sorted heaviest first, dealt to the CTAs in snake order (rounds of
    // gridDim.x alternate direction) so that every CTA's total is close to the mean
    const int sorted = snake_sorted(it, p.n_items);
    qp = p.n_pairs - 1 - sorted / bh_count;
    w.bh = sorted % bh_count;
  } else {  // head-major: CTAs working at the same time share a head's K/V in L2
    w.bh = it / p.n_pairs;
    qp = it % p.n_pairs;
  }
  w.b = w.bh / p.Hkv;
  w.kvh = w.bh % p.Hkv;
  const int S_b = item_keys<PAGED>(p, w.b);
  const int shift = S_b - p.T;  // bottom-right: query i sits at key position i + shift
  const int lo = split_j0<SPLIT>(p, it) * bn;  // first key of this item's range
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int first = (2 * qp + t) * p.rows_per_head;
    int kv_end = 0;
    if (first < p.T) {
      kv_end = S_b;
      if (p.causal) kv_end = min(S_b, min(first + p.rows_per_head, p.T) - 1 + shift + 1);
    }
    if (SPLIT) kv_end = min(kv_end, lo + p.split_tiles * bn);
    w.p0[t] = first;
    w.nj[t] = kv_end > lo ? (kv_end - lo + bn - 1) / bn : 0;
  }
  return w;
}

template <int D, bool PAGED, bool SPLIT>
__global__ void __launch_bounds__(384, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const PfParams p) {
  using C = PfCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  PfBars* bars = reinterpret_cast<PfBars*>(smem + C::OFF_BAR);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // A launch that follows this one on the stream as a programmatic dependent (the next
  // call of this kernel) may start its CTAs as SMs free up; it reads nothing of ours
  // before its griddepcontrol.wait, which returns only once this grid has completed and
  // its stores are visible. The key split is followed by its merge, whose thousands of
  // small blocks would only sit waiting on the SMs; it launches at this grid's end.
  if constexpr (!SPLIT) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 128);
      mbar_init(&bars->pv_done[s], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::MMA_WARP) tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
  // This grid may itself have started before the work ahead of it on the stream
  // completed (it launches as a programmatic dependent): nothing global is read or
  // written before that work is complete and visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // paged: rank the sequences by key count, longest first (ties by index)
  int* order_smem = reinterpret_cast<int*>(smem + C::OFF_ORDER);
  const int* order = nullptr;
  if (PAGED && p.B <= C::MAX_RANKED) {
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
      const int sb = item_keys<PAGED>(p, b);
      int rank = 0;
      for (int b2 = 0; b2 < p.B; ++b2) {
        const int s2 = item_keys<PAGED>(p, b2);
        rank += (s2 > sb || (s2 == sb && b2 < b)) ? 1 : 0;
      }
      order_smem[rank] = b;
    }
    order = order_smem;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;
  const uint64_t tmo = p.timeout_ns;
  const uint64_t tmo_unwind = unwind_timeout(tmo);  // copies landing, MMAs draining

  const int shift_all = p.S - p.T;  // contiguous: bottom-right alignment, one shift for every item

  auto fail = [&](unsigned site) {
    record_error(p.err, FA_ERR_TIMEOUT, site);
    *abort_flag = 1;
  };

  if (warp >= 8) {
    // setmaxnreg is issued at the head of each role's branch so that the
    // register budget it sets governs all of that role's code
    warpgroup_reg_dealloc<C::AUX_REGS>();
  if (warp == C::PRODUCER_WARP) {
    // ======================= TMA producer =======================
    // Contiguous K/V: one lane does everything. Paged K/V: a key tile is 16 page
    // boxes per operand, so the whole warp runs the loop (its waits are uniform:
    // every lane polls the same barrier in one instruction), lanes 0-7 hold the
    // tile's table entries, and one box per lane is issued after lane 0 has armed
    // the barrier.
    if (PAGED || lane == 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
      }
      uint32_t g = 0;  // key tiles loaded so far, over all items (ring position)
      int item_i = 0;
      uint32_t q_loads = 0;  // Q loads issued (q_full phases)
      for (int it = blockIdx.x; it < p.n_items && !*abort_flag; it += gridDim.x, ++item_i) {
        const PfItem w = pf_item<PAGED, SPLIT>(p, it, C::BN, order);
        const int nj = max(w.nj[0], w.nj[1]);
        // Q of the previous item stays in smem until its last S has been computed
        if (item_i > 0 && !mbar_wait(&bars->q_empty, (item_i - 1) & 1, tmo, abort_flag)) {
          fail(SITE_PF_PRODUCER);
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->q_full, C::QT * C::Q_BYTES);
          for (int t = 0; t < 2; ++t)
            for (int c = 0; c < C::KCH; ++c)
              tma_load_4d(sQ + t * C::Q_BYTES + c * C::CHUNK_BYTES, &tmQ, &bars->q_full, c * 64, w.p0[t],
                          w.kvh * p.g, w.b);
        }
        ++q_loads;
        // paged: the 128 keys of tile j are pages 8j .. 8j+7 of the sequence; pages past
        // its end are not loaded (their K is masked, their V zeroed before use). Lane
        // i < 8 holds the entry of page 8j + i; the next tile's are fetched while this
        // tile is issued.
        const int j0 = split_j0<SPLIT>(p, it);  // first key tile of the item's range
        const int* trow = PAGED ? p.block_table + static_cast<size_t>(w.b) * p.max_pages : nullptr;
        const int n_pages = (item_keys<PAGED>(p, w.b) + 15) >> 4;
        auto fetch = [&](int jt) -> int {
          const int pg = jt * 8 + lane;
          return (PAGED && lane < 8 && jt < nj && pg < n_pages) ? __ldg(trow + pg) : -1;
        };
        int ent_next = PAGED ? fetch(0) : -1;
        for (int j = 0; j < nj; ++j, ++g) {
          const int s = g % C::STAGES;
          const uint32_t u = g / C::STAGES;
          int npg = 8;  // pages of this tile that are loaded
          int ent = -1;
          if (PAGED) {
            ent = ent_next;
            ent_next = fetch(j + 1);
            npg = min(8, n_pages - j * 8);
            if (lane < npg && (ent < 0 || ent >= p.num_pages)) {
              // never dereferenced: the tile still receives the bytes it expects,
              // from page 0, and the sequence's output is undefined
              record_error(p.err, FA_ERR_BOUNDS, SITE_PF_TABLE);
              ent = 0;
            }
          }
          const uint32_t tile_bytes = PAGED ? static_cast<uint32_t>(npg) * 16 * 128 * C::KCH : C::KV_BYTES;
          // paged: lane L issues the box of page L / KCH, d-chunk L % KCH
          const int pi = lane / C::KCH, pc = lane % C::KCH;
          const int pe = PAGED ? __shfl_sync(0xffffffffu, ent, pi & 7) : 0;
          if (g >= C::STAGES && !mbar_wait(&bars->k_empty[s], (u - 1) & 1, tmo, abort_flag)) {
            fail(SITE_PF_PRODUCER);
            break;
          }
          if (PAGED) {
            if (lane == 0) mbar_arrive_expect_tx(&bars->k_full[s], tile_bytes);
            __syncwarp();
            if (pi < npg)
              tma_load_3d(sK + s * C::KV_BYTES + pc * C::CHUNK_BYTES + pi * 16 * 128, &tmK, &bars->k_full[s],
                          pc * 64, w.kvh, pe * 16);
          } else {
            mbar_arrive_expect_tx(&bars->k_full[s], tile_bytes);
            for (int c = 0; c < C::KCH; ++c)
              tma_load_3d(sK + s * C::KV_BYTES + c * C::CHUNK_BYTES, &tmK, &bars->k_full[s], c * 64, (j0 + j) * C::BN,
                          w.bh);
          }
          if (g >= C::STAGES && !mbar_wait(&bars->v_empty[s], (u - 1) & 1, tmo, abort_flag)) {
            fail(SITE_PF_PRODUCER);
            mbar_wait(&bars->k_full[s], u & 1, tmo_unwind);  // K was issued: let it land
            break;
          }
          if (PAGED) {
            if (lane == 0) mbar_arrive_expect_tx(&bars->v_full[s], tile_bytes);
            __syncwarp();
            if (pi < npg)
              tma_load_3d(sV + s * C::KV_BYTES + pc * C::CHUNK_BYTES + pi * 16 * 128, &tmV, &bars->v_full[s],
                          pc * 64, w.kvh, pe * 16);
          } else {
            mbar_arrive_expect_tx(&bars->v_full[s], tile_bytes);
            for (int c = 0; c < C::KCH; ++c)
              tma_load_3d(sV + s * C::KV_BYTES + c * C::CHUNK_BYTES, &tmV, &bars->v_full[s], c * 64, (j0 + j) * C::BN,
                          w.bh);
          }
        }
      }
      if (*abort_flag) {
        // copies still in flight must complete before the CTA exits
        if (q_loads > 0) mbar_wait(&bars->q_full, (q_loads - 1) & 1, tmo_unwind);
        for (uint32_t x = g > C::STAGES ? g - C::STAGES : 0; x < g; ++x) {
          mbar_wait(&bars->k_full[x % C::STAGES], (x / C::STAGES) & 1, tmo_unwind);
          mbar_wait(&bars->v_full[x % C::STAGES], (x / C::STAGES) & 1, tmo_unwind);
        }
      }
    }
  } else if (warp == C::MMA_WARP) {
    // ======================= MMA issuer =======================
    // The whole warp runs the loop (waits, descriptors, loop control stay
    // warp-uniform); one elected lane issues each MMA and commit.
    const bool leader = elect_one();
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, C::BN, 0, 0);  // A = Q (K-major), B = K (K-major)
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);      // A = P (TMEM), B = V (MN-major)
    // descriptors of the operand bases; an MMA adds its (compile-time) byte offset >> 4
    // to the start-address field, which never carries out of its 14 bits (smem < 256 KB)
    const uint64_t dQ = smem_desc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dK = smem_desc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t dV = smem_desc_sw128(smem_u32(sV), C::CHUNK_BYTES, 1024);
    // S_t = Q_t K^T (K in ring stage st) into tile t's S/P columns
    auto qk = [=](int t, int st) {
      const uint64_t a0 = dQ + static_cast<uint64_t>((t * C::Q_BYTES) >> 4);
      const uint64_t b0 = dK + static_cast<uint64_t>((st * C::KV_BYTES) >> 4);
      const uint32_t dS = tmem + t * C::TILE_COLS;
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // 16 elements of d per MMA: chunk kk/4, 32-byte step inside the 128-byte swizzle row
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4);
          tc_mma_ss(dS, a0 + off, b0 + off, idesc_qk, kk > 0 ? 1u : 0u);
        }
      }
    };
    // O_t (+)= P_t V (V in ring stage st): P from TMEM (8 columns = 16 keys per MMA),
    // V MN-major from smem; the first key tile of an item overwrites O
    auto pv = [=](int t, int st, bool first) {
      const uint64_t b0 = dV + static_cast<uint64_t>((st * C::KV_BYTES) >> 4);
      const uint32_t dO = tmem + t * C::TILE_COLS + C::O_OFF;
      const uint32_t aP = tmem + t * C::TILE_COLS;
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          tc_mma_ts(dO, aP + kk * 8, b0 + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv,
                    (!first || kk > 0) ? 1u : 0u);
      }
    };
    auto commit = [=](uint64_t* bar) {
      if (leader) tc_commit(bar);
    };
    // every lane polls the same barrier and the same timer in the same
    // instruction, so the outcome is warp-uniform without a vote
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool { return mbar_wait(bar, parity, tmo, abort_flag); };
    bool ok = true;
    uint32_t g = 0;                // key tiles consumed so far, over all items (ring position)
    uint32_t pph0 = 0, pph1 = 0;   // p_full phase parity of tile 0 / 1
    int item_i = 0;
    for (int it = blockIdx.x; ok && it < p.n_items; it += gridDim.x, ++item_i) {
      const PfItem w = pf_item<PAGED, SPLIT>(p, it, C::BN, order);
      const int nj0 = w.nj[0], nj1 = w.nj[1];
      const int nj = max(nj0, nj1);
      if (!wwait(&bars->q_full, item_i & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (nj == 0) {
        if (leader) mbar_arrive(&bars->q_empty);  // nothing read Q
        continue;
      }
      if (!wwait(&bars->k_full[g & 1], (g >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (nj0 > 0) {
        qk(0, g & 1);
        commit(&bars->s_full[0]);
      }
      if (nj1 > 0) {
        qk(1, g & 1);
        commit(&bars->s_full[1]);
      }
      commit(&bars->k_empty[g & 1]);
      if (nj == 1) commit(&bars->q_empty);  // that was this item's last S
      static_assert(C::STAGES == 2, "the issue loop below indexes a two-stage K/V ring");
      // K/V ring of two stages: key tile x sits in stage x & 1, phase (x >> 1) & 1.
      // The first PV of an item overwrites O_t; the softmax threads read O_t out
      // for the previous item before they publish this item's first P_t, so the
      // P wait orders it. A rescale of O at step j needs PV_t(j-1) finished, which
      // the S_t(j) commit (issued after it) implies, so pv_done is per item.
      for (int j = 0; j < nj; ++j) {
        const uint32_t gj = g + j;
        const int s = gj & 1;                       // V_j (and K_j)
        const uint32_t vph = (gj >> 1) & 1;
        const int s1 = s ^ 1;                       // K_{j+1}
        const uint32_t kph1 = ((gj + 1) >> 1) & 1;
        bool k_ready = false;
        // ---- tile 0
        if (j < nj0) {
          if (!wwait(&bars->p_full[0], pph0) || !wwait(&bars->v_full[s], vph)) {
            ok = false;
            break;
          }
          pph0 ^= 1;
          tc_fence_after();
          pv(0, s, j == 0);
          if (j + 1 == nj0) commit(&bars->pv_done[0]);
          if (j >= nj1) commit(&bars->v_empty[s]);  // tile 1 does not read V_j
          // the next S of this tile overwrites the columns P_0 is read from; MMAs
          // issued by one thread execute in order, so it is queued right behind
          if (j + 1 < nj0) {
            if (!wwait(&bars->k_full[s1], kph1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            k_ready = true;
            qk(0, s1);
            commit(&bars->s_full[0]);
          }
        }
        // ---- tile 1
        if (j < nj1) {
          if (!wwait(&bars->p_full[1], pph1) || (j >= nj0 && !wwait(&bars->v_full[s], vph))) {
            ok = false;
            break;
          }
          pph1 ^= 1;
          tc_fence_after();
          pv(1, s, j == 0);
          if (j + 1 == nj1) commit(&bars->pv_done[1]);
          commit(&bars->v_empty[s]);
          if (j + 1 < nj1) {
            if (!k_ready) {
              if (!wwait(&bars->k_full[s1], kph1)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            qk(1, s1);
            commit(&bars->s_full[1]);
          }
        }
        if (j + 1 < nj) commit(&bars->k_empty[s1]);
        if (j + 2 == nj) commit(&bars->q_empty);  // the item's last S was just issued
      }
      g += nj;
    }
    if (!ok && leader) fail(SITE_PF_MMA);
    // every MMA issued must finish before TMEM is released
    commit(&bars->drain);
    mbar_wait(&bars->drain, 0, tmo_unwind);
  }
  } else {
    // ======================= softmax: warps 0-3 (tile 0), 4-7 (tile 1) =======================
    warpgroup_reg_alloc<C::SOFTMAX_REGS>();
    const int t = warp >> 2;
    const int r = threadIdx.x & 127;  // row of the tile == TMEM lane
    const int h_local = r / p.rows_per_head;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * C::TILE_COLS;
    const uint32_t tO = tS + C::O_OFF;
    const float c = p.c;
    const float2 c2 = make_float2(c, c);
    // m: the row's reference max, in units of log2 (scores times c); l: the running
    // sum of 2^(s*c - m); O in TMEM holds the matching unnormalised sum of P V.
    // The reference is raised (and l, O rescaled by 2^(m_old - m_new)) only when
    // the row max climbs more than kRescaleSlack above it; below that the
    // exponentials are taken against the slightly stale reference and stay
    // <= 2^kRescaleSlack. Every term then carries the same constant factor,
    // which O / l cancels, so the result is the same softmax.
    constexpr float kRescaleSlack = 8.f;
    bool ok = true;
    // waits are warp-collective: the warp leaves together, so the .sync.aligned
    // tcgen05 loads and the votes below always see all 32 lanes
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool w = mbar_wait(bar, parity, tmo, abort_flag);
      return __all_sync(0xffffffffu, w);
    };
    uint32_t cnt = 0;   // key tiles of this query tile done so far, over all items (s_full phases)
    uint32_t ecnt = 0;  // items of this query tile with at least one key tile (pv_done phases)
    uint32_t gkv = 0;   // K/V ring position at the start of the item (paged V tail zeroing)
    for (int it = blockIdx.x; ok && it < p.n_items; it += gridDim.x) {
      const PfItem w = pf_item<PAGED, SPLIT>(p, it, C::BN, order);
      const int S_item = item_keys<PAGED>(p, w.b);  // keys of this item's sequence
      const int shift = PAGED ? S_item - p.T : shift_all;  // bottom-right: row i sees keys j <= i + shift
      const int nj_item = max(w.nj[0], w.nj[1]);
      // paged: V rows past the sequence end in its last key tile hold whatever the pool
      // (or an earlier tile) left there, possibly NaN, and a zero weight would not cancel
      // a NaN. The tile that issues the first PV on that key tile zeroes them first.
      const bool v_tail_owner = PAGED && nj_item > 0 && nj_item * C::BN > S_item && t == (w.nj[0] == nj_item ? 0 : 1);
      // selects, not a runtime index into w (which would put w in local memory)
      const int my_nj = t ? w.nj[1] : w.nj[0];
      const int my_p0 = t ? w.p0[1] : w.p0[0];
      const int pos = my_p0 + (r % p.rows_per_head);
      const bool row_valid = pos < p.T;
      const int vis_last = pos + shift;  // causal: last visible key of this row
      float m = -INFINITY;
      float l = 0.f;   // sum of the unrounded p: the lse's sum
      float lc = 0.f;  // per tile, bf16(p_top) - p_top of its largest p, rescaled like l

      for (int j = 0; j < my_nj; ++j, ++cnt) {
        if (!wwait(&bars->s_full[t], cnt & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // S row: four 32-column loads in flight, one wait
        uint32_t raw[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, raw[cc]);
        tmem_ld_wait();
        float s[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(raw[i >> 5][i & 31]);

        const int key0 = (split_j0<SPLIT>(p, it) + j) * C::BN;
        const bool need_mask = (key0 + C::BN > S_item) || (p.causal && key0 + C::BN - 1 > my_p0 + shift);
        if (need_mask) {
          const int lim = (p.causal ? min(S_item - 1, vis_last) : S_item - 1) - key0;
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i > lim) s[i] = -INFINITY;
        }
        // row max: eight independent three-input chains, then a short tree
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float a = fmax3(s[16 * k], s[16 * k + 1], s[16 * k + 2]);
#pragma unroll
          for (int i = 3; i < 15; i += 2) a = fmax3(a, s[16 * k + i], s[16 * k + i + 1]);
          mx8[k] = fmaxf(a, s[16 * k + 15]);
        }
        const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        const float m_tile = mx * c;
        const float m_new = (m_tile > m + kRescaleSlack) ? m_tile : m;  // m = -inf: first visible key sets it
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx(m - m_use);  // 1 if the reference is kept; 0 while nothing was seen
        // The tile's largest p, computed exactly as the loop below computes it for
        // that key, and its rounding to the bf16 the P V product consumes. Against
        // a stale reference the largest p is up to 2^kRescaleSlack, not exactly 1,
        // so its bf16 rounding would leave a near-one-hot row's O off by 2^-9
        // relative; O's normaliser l + lc counts that term as P V sees it.
        const float p_top = ex2_approx(fmaf(mx, c, -m_use));
        const float p_top_err = __bfloat162float(__float2bfloat16_rn(p_top)) - p_top;
        // p = 2^(s*c - m): packed FFMA, MUFU ex2, bf16 pairs stored over S, 32 columns at a time
        const float2 nm2 = make_float2(-m_use, -m_use);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int e = cc * 32 + 2 * i;
            const float2 x = ffma2(make_float2(s[e], s[e + 1]), c2, nm2);
            const float2 ev = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            acc[i & 3] = fadd2(acc[i & 3], ev);
            pk[i] = pack_bf16x2(ev.x, ev.y);
          }
          tmem_st16(tS + cc * 16, pk);  // keys 32cc .. 32cc+31 -> columns 16cc .. 16cc+15
        }
        const float2 a01 = fadd2(acc[0], acc[1]);
        const float2 a23 = fadd2(acc[2], acc[3]);
        const float2 at = fadd2(a01, a23);
        l = fmaf(l, alpha, at.x + at.y);
        lc = fmaf(lc, alpha, p_top_err);
        m = m_new;

        // O is rescaled only when the max of some row of this warp rose; that
        // needs PV_t(j-1) finished (it accumulates into O), which S_t(j) being
        // complete already implies: its commit was issued after that PV
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
          for (int cc = 0; cc < D / 32; cc += 2) {
            uint32_t o0[32], o1[32];
            tmem_ld32(tO + cc * 32, o0);
            tmem_ld32(tO + cc * 32 + 32, o1);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float2 v0 = fmul2(make_float2(__uint_as_float(o0[i]), __uint_as_float(o0[i + 1])), al2);
              float2 v1 = fmul2(make_float2(__uint_as_float(o1[i]), __uint_as_float(o1[i + 1])), al2);
              o0[i] = __float_as_uint(v0.x);
              o0[i + 1] = __float_as_uint(v0.y);
              o1[i] = __float_as_uint(v1.x);
              o1[i + 1] = __float_as_uint(v1.y);
            }
            tmem_st32(tO + cc * 32, o0);
            tmem_st32(tO + cc * 32 + 32, o1);
          }
        }
        if (v_tail_owner && j + 1 == nj_item) {
          // zero V rows S_item - key0 .. 127 of this key tile once its copy has landed,
          // then make the generic stores visible to the tensor core's reads
          const uint32_t x = gkv + j;
          if (!wwait(&bars->v_full[x % C::STAGES], (x / C::STAGES) & 1)) {
            ok = false;
            break;
          }
          uint8_t* vt = sV + (x % C::STAGES) * C::KV_BYTES;
          const int r0 = S_item - key0;
          for (int idx = r; idx < (C::BN - r0) * C::KCH * 8; idx += 128) {
            const int row = r0 + idx / (C::KCH * 8);
            const int rem = idx % (C::KCH * 8);
            *reinterpret_cast<uint4*>(vt + (rem >> 3) * C::CHUNK_BYTES + row * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_async_smem();
        }
        tmem_st_wait();  // P (and O) stores complete before the MMA may read them
        tc_fence_before();
        mbar_arrive(&bars->p_full[t]);
      }
      gkv += nj_item;

      // ---- epilogue: O / l -> bf16, lse = ln2 * (m + log2 l)
      if (ok && my_nj > 0) {
        if (!wwait(&bars->pv_done[t], ecnt & 1)) ok = false;
        ++ecnt;
        tc_fence_after();
      }
      if (!ok) fail(SITE_PF_SOFTMAX);
      const int h = w.kvh * p.g + h_local;
      const size_t row_index = (static_cast<size_t>(w.b) * p.Hq + h) * p.T + pos;
      __nv_bfloat16* orow = p.o + row_index * D;
      if (ok) {
        const float inv_l = l > 0.f ? 1.f / (l + lc) : 0.f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          if (my_nj > 0) {
            tmem_ld32(tO + cc * 32, o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
          }
          if (SPLIT) {
            // the range's normalised partial, fp32, for the LSE merge
            if (row_valid) {
              float* prow = p.o_part + (static_cast<size_t>(it % p.num_splits) * p.B * p.Hq * p.T + row_index) * D;
#pragma unroll
              for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4*>(prow + cc * 32 + 4 * q) =
                    make_float4(__uint_as_float(o[4 * q + 0]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                                __uint_as_float(o[4 * q + 2]) * inv_l, __uint_as_float(o[4 * q + 3]) * inv_l);
            }
          } else if (row_valid) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv_l, __uint_as_float(o[8 * q + 1]) * inv_l);
              v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv_l, __uint_as_float(o[8 * q + 3]) * inv_l);
              v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv_l, __uint_as_float(o[8 * q + 5]) * inv_l);
              v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv_l, __uint_as_float(o[8 * q + 7]) * inv_l);
              *reinterpret_cast<uint4*>(orow + cc * 32 + 8 * q) = v;
            }
          }
        }
        const float lse_v = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        if (SPLIT) {
          if (row_valid) p.lse_part[static_cast<size_t>(it % p.num_splits) * p.B * p.Hq * p.T + row_index] = lse_v;
        } else if (row_valid && p.lse) {
          p.lse[row_index] = lse_v;
        }
      }
      // O_t has been read out (the loads above completed); these threads arrive on
      // p_full for the next item only after this, so the MMA warp's wait for that P
      // also orders the next item's first PV (which overwrites O_t) after these reads
      if (ok && my_nj > 0) tc_fence_before();
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
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();  // defined in api.cu
int device_sm_count();              // defined in api.cu

template <int D, bool PAGED, bool SPLIT = false>
static int launch_pf(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PfParams& p, int grid,
                     cudaStream_t stream) {
  auto kfn = prefill_tc_kernel<D, PAGED, SPLIT>;
  const int smem = PAGED ? PfCfg<D>::SMEM_PAGED : PfCfg<D>::SMEM;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return FA_ERR_CUDA;
  // a programmatic dependent of the previous launch on the stream: the CTAs' setup
  // (barriers, TMEM) overlaps that launch's tail; the kernel waits before any global access
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(PfCfg<D>::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kfn, tq, tk, tv, p) != cudaSuccess) return FA_ERR_CUDA;
  return launch_status();
}

// Contiguous K/V ([B][Hkv][S][d]) when block_table is null; otherwise `k`/`v` are
// pools [num_pages][16][Hkv][d] shared through block_table [B][max_pages], with
// seqlens [B] keys per sequence (S is then unused). num_splits > 1 (contiguous
// only): the keys are cut into num_splits ranges of whole 128-key tiles and the
// kernel writes normalised fp32 partials to o_part / lse_part (layout of
// fa_decode_workspace_bytes) instead of o / lse; the caller merges them.
int launch_prefill_tc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                      int T, int S, int d, float scale, int causal, cudaStream_t stream, unsigned* err,
                      unsigned long long timeout_ns, const int* block_table, const int* seqlens, int max_pages,
                      int num_pages, int num_splits, float* o_part, float* lse_part) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return FA_ERR_CUDA;
  const bool paged = block_table != nullptr;
  const int g = Hq / Hkv;
  const int rows_per_head = 128 / g;
  CUtensorMap tq, tk, tv;
  {
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)Hq, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)T * d * 2, (cuuint64_t)Hq * T * d * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)rows_per_head, (cuuint32_t)g, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FA_ERR_CUDA;
  }
  for (int w = 0; w < 2; ++w) {
    cuuint64_t dims[3];
    cuuint64_t strides[2];
    cuuint32_t box[3];
    if (!paged) {
      // 128 keys of one (batch, KV head) per box
      dims[0] = d; dims[1] = S; dims[2] = static_cast<cuuint64_t>(B) * Hkv;
      strides[0] = static_cast<cuuint64_t>(d) * 2;
      strides[1] = static_cast<cuuint64_t>(S) * d * 2;
      box[0] = 64; box[1] = 128; box[2] = 1;
    } else {
      // one 16-token page of one KV head per box
      dims[0] = d; dims[1] = Hkv; dims[2] = static_cast<cuuint64_t>(num_pages) * 16;
      strides[0] = static_cast<cuuint64_t>(d) * 2;
      strides[1] = static_cast<cuuint64_t>(Hkv) * d * 2;
      box[0] = 64; box[1] = 1; box[2] = 16;
    }
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(w == 0 ? &tk : &tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w == 0 ? k : v), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FA_ERR_CUDA;
  }
  PfParams p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.T = T;
  p.S = paged ? max_pages * 16 : S;
  p.g = g;
  p.rows_per_head = rows_per_head;
  p.n_qtiles = (T + rows_per_head - 1) / rows_per_head;
  p.n_pairs = (p.n_qtiles + 1) / 2;
  p.causal = causal;
  p.c = scale * kLog2e;
  p.err = err;
  p.timeout_ns = timeout_ns;
  p.block_table = block_table;
  p.seqlens = seqlens;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  const bool split = num_splits > 1 && !paged;
  p.num_splits = split ? num_splits : 1;
  // ranges of whole key tiles: no tile is shared by two ranges
  p.split_tiles = split ? ((S + 127) / 128 + num_splits - 1) / num_splits : 0;
  p.o_part = o_part;
  p.lse_part = lse_part;
  const long long items = static_cast<long long>(p.n_pairs) * B * Hkv * p.num_splits;
  if (items > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  p.n_items = static_cast<int>(items);
  // persistent: one CTA per SM, each takes items blockIdx.x, blockIdx.x + grid, ...
  const int sms = device_sm_count();
  if (sms <= 0) return FA_ERR_CUDA;
  const int grid = items < sms ? static_cast<int>(items) : sms;
  if (d == 128) {
    if (paged) return launch_pf<128, true>(tq, tk, tv, p, grid, stream);
    return split ? launch_pf<128, false, true>(tq, tk, tv, p, grid, stream)
                 : launch_pf<128, false>(tq, tk, tv, p, grid, stream);
  }
  if (paged) return launch_pf<64, true>(tq, tk, tv, p, grid, stream);
  return split ? launch_pf<64, false, true>(tq, tk, tv, p, grid, stream) : launch_pf<64, false>(tq, tk, tv, p, grid, stream);
}

}  // namespace fa
