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
//   * one CTA per (batch, KV head, tile of BM = 128 query rows). With GQA the
//     g query heads of a group are stacked as rows of one tile (128/g
//     positions x g heads), so every K/V tile is loaded once per group ("GQA
//     loads KV once per group"). A 4-D TMA box {64, 128/g, g, 1} over Q
//     [B][Hq][T][d] builds the stacked tile directly.
//   * warp 4 (one elected thread): TMA producer. Q once, then K_j and V_j
//     into a 2-stage ring of 128-byte-swizzled shared-memory tiles; separate
//     full/empty mbarriers for K and V so K can be refilled as soon as
//     S_j = Q K_j^T has consumed it.
//   * warp 5: allocates 512 TMEM columns; one thread issues tcgen05.mma.
//     S_j (fp32, 128 columns) goes to one of two TMEM buffers so S_{j+1} is
//     computed while the softmax works on S_j; O (fp32, d columns) stays in
//     TMEM for the whole row of tiles.
//   * warps 0-3 (128 threads, thread r = row r = TMEM lane r): softmax.
//     tcgen05.ld of S_j, row max, p = 2^(s*c - m) with c = scale*log2(e)
//     folded into one FFMA, P packed to bf16 and written to a swizzled smem
//     tile (the A operand of O += P V_j). O is rescaled in TMEM only when
//     the max of some row of the warp rose.
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
  static constexpr int BM = 128;           // query rows per tile (TMEM lanes)
  static constexpr int BN = 128;           // keys per K/V tile
  static constexpr int KCH = D / 64;       // 64-element (128-byte) chunks along d
  static constexpr int STAGES = 2;         // K/V ring depth
  static constexpr int CHUNK_BYTES = 128 * 128;  // one 128-row x 128-byte swizzled chunk
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int P_BYTES = BM * BN * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_P = OFF_V + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;  // + slack to align the base to 1024
  static constexpr int TMEM_COLS = 512;
  static constexpr int S_COL1 = 128;  // S buffer b lives at column b * S_COL1
  static constexpr int O_COL = 256;
  static constexpr int THREADS = 192;
};

struct PfParams {
  __nv_bfloat16* o;
  float* lse;
  int B, Hq, Hkv, T, S;
  int g;              // query heads per KV head
  int rows_per_head;  // 128 / g query positions per tile
  int n_qtiles;       // ceil(T / rows_per_head)
  int causal;
  float c;            // scale * log2(e)
  unsigned* err;
  unsigned long long timeout_ns;
};

struct PfBars {
  uint64_t q_full;
  uint64_t k_full[2], v_full[2], k_empty[2], v_empty[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, o_done, drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const PfParams p) {
  using C = PfCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sP = smem + C::OFF_P;
  PfBars* bars = reinterpret_cast<PfBars*>(smem + C::OFF_BAR);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (b, kv head, query tile); causal runs heaviest tiles first
  const int bh_count = p.B * p.Hkv;
  int qt, bh;
  if (p.causal) {
    qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x) / bh_count;
    bh = static_cast<int>(blockIdx.x) % bh_count;
  } else {
    bh = static_cast<int>(blockIdx.x) / p.n_qtiles;
    qt = static_cast<int>(blockIdx.x) % p.n_qtiles;
  }
  const int b = bh / p.Hkv;
  const int kvh = bh % p.Hkv;
  const int p0 = qt * p.rows_per_head;  // first query position of the tile
  const int shift = p.S - p.T;           // bottom-right alignment: row i sees keys j <= i + shift
  int kv_end = p.S;
  if (p.causal) {
    const int last_pos = min(p0 + p.rows_per_head, p.T) - 1;
    kv_end = min(p.S, last_pos + shift + 1);
  }
  const int nj = kv_end > 0 ? (kv_end + C::BN - 1) / C::BN : 0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], 128);
    }
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;
  const uint64_t tmo = p.timeout_ns;

  auto fail = [&](unsigned site) {
    record_error(p.err, FA_ERR_TIMEOUT, site);
    *abort_flag = 1;
  };

  if (warp == 4) {
    // ======================= TMA producer =======================
    if (lane == 0 && nj > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(&bars->q_full, C::Q_BYTES);
      for (int c = 0; c < C::KCH; ++c)
        tma_load_4d(sQ + c * C::CHUNK_BYTES, &tmQ, &bars->q_full, c * 64, p0, kvh * p.g, b);
      int issued = 0;
      for (int j = 0; j < nj; ++j) {
        const int s = j % C::STAGES;
        const uint32_t u = j / C::STAGES;
        if (j >= C::STAGES && !mbar_wait(&bars->k_empty[s], (u - 1) & 1, tmo, abort_flag)) {
          fail(SITE_PF_PRODUCER);
          break;
        }
        mbar_arrive_expect_tx(&bars->k_full[s], C::KV_BYTES);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(sK + s * C::KV_BYTES + c * C::CHUNK_BYTES, &tmK, &bars->k_full[s], c * 64, j * C::BN, bh);
        if (j >= C::STAGES && !mbar_wait(&bars->v_empty[s], (u - 1) & 1, tmo, abort_flag)) {
          fail(SITE_PF_PRODUCER);
          // K_j was issued: let its copy land before the CTA's smem goes away
          mbar_wait(&bars->k_full[s], u & 1, tmo);
          break;
        }
        mbar_arrive_expect_tx(&bars->v_full[s], C::KV_BYTES);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(sV + s * C::KV_BYTES + c * C::CHUNK_BYTES, &tmV, &bars->v_full[s], c * 64, j * C::BN, bh);
        issued = j + 1;
      }
      if (*abort_flag) {
        // drain: copies still in flight must complete before the CTA exits
        mbar_wait(&bars->q_full, 0, tmo);
        for (int j = max(0, issued - C::STAGES); j < issued; ++j) {
          mbar_wait(&bars->k_full[j % C::STAGES], (j / C::STAGES) & 1, tmo);
          mbar_wait(&bars->v_full[j % C::STAGES], (j / C::STAGES) & 1, tmo);
        }
      }
    }
  } else if (warp == 5) {
    // ======================= MMA issuer =======================
    if (lane == 0 && nj > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, C::BN, 0, 0);  // A = Q (K-major), B = K (K-major)
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);      // A = P (K-major), B = V (MN-major)
      const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV), sPa = smem_u32(sP);
      bool ok = mbar_wait(&bars->q_full, 0, tmo, abort_flag);
      auto issue_qk = [&](int j) -> bool {
        const int s = j % C::STAGES;
        if (!mbar_wait(&bars->k_full[s], (j / C::STAGES) & 1, tmo, abort_flag)) return false;
        if (j >= 2 && !mbar_wait(&bars->s_free[j & 1], ((j >> 1) & 1) ^ 1, tmo, abort_flag)) return false;
        tc_fence_after();
        const uint32_t kbase = sKa + s * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // 16 elements of d per MMA: chunk kk/4, 32-byte step inside the 128-byte swizzle row
          const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          tc_mma_ss(tmem + (j & 1) * C::S_COL1, smem_desc_sw128(sQa + off, 16, 1024),
                    smem_desc_sw128(kbase + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(&bars->k_empty[s]);
        tc_commit(&bars->s_full[j & 1]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int j = 0; ok && j < nj; ++j) {
        if (j + 1 < nj && !issue_qk(j + 1)) {
          ok = false;
          break;
        }
        const int s = j % C::STAGES;
        if (!mbar_wait(&bars->p_full, j & 1, tmo, abort_flag) ||
            !mbar_wait(&bars->v_full[s], (j / C::STAGES) & 1, tmo, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t vbase = sVa + s * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          // A = P: 16 keys per MMA (chunk kk/4 of the swizzled P tile);
          // B = V, MN-major: 16 keys = two 8-row groups of 1024 bytes; LBO steps over d chunks
          const uint32_t poff = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          tc_mma_ss(tmem + C::O_COL, smem_desc_sw128(sPa + poff, 16, 1024),
                    smem_desc_sw128(vbase + kk * 2048, C::CHUNK_BYTES, 1024), idesc_pv,
                    (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&bars->v_empty[s]);
        tc_commit(&bars->o_done);
      }
      if (!ok) {
        fail(SITE_PF_MMA);
        // every MMA issued so far must finish before TMEM is released
        tc_commit(&bars->drain);
        mbar_wait(&bars->drain, 0, tmo);
      }
    }
  } else {
    // ======================= softmax: warps 0-3, one row per thread =======================
    const int r = threadIdx.x;  // row of the tile == TMEM lane
    const int h_local = r / p.rows_per_head;
    const int pos = p0 + (r % p.rows_per_head);
    const bool row_valid = pos < p.T;
    const int vis_last = pos + shift;  // causal: last visible key of this row
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float c = p.c;
    float m = -INFINITY;  // running max, in units of log2 (scores times c)
    float l = 0.f;        // running sum of 2^(s*c - m)
    bool ok = true;
    // waits are warp-collective: the warp leaves together, so the .sync.aligned
    // tcgen05 loads and the votes below always see all 32 lanes
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool w = mbar_wait(bar, parity, tmo, abort_flag);
      return __all_sync(0xffffffffu, w);
    };
    uint8_t* prow = sP + r * 128;
    const int rsw = r & 7;

    for (int j = 0; j < nj; ++j) {
      const int sb = j & 1;
      if (!wwait(&bars->s_full[sb], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t raw[32];
        tmem_ld32(tmem + lane_base + sb * C::S_COL1 + cc * 32, raw);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[cc * 32 + i] = __uint_as_float(raw[i]);
      }
      tc_fence_before();
      mbar_arrive(&bars->s_free[sb]);

      const int key0 = j * C::BN;
      const bool need_mask = (key0 + C::BN > p.S) || (p.causal && key0 + C::BN - 1 > p0 + shift);
      if (need_mask) {
        const int lim = p.causal ? min(p.S - 1, vis_last) : p.S - 1;
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (key0 + i > lim) s[i] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int i = 1; i < 128; ++i) mx = fmaxf(mx, s[i]);
      const float m_new = fmaxf(m, mx * c);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m - m_use);  // 0 while nothing was seen (m = -inf)
      float rs = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float e0 = ex2_approx(fmaf(s[2 * i], c, -m_use));
        const float e1 = ex2_approx(fmaf(s[2 * i + 1], c, -m_use));
        rs += e0 + e1;
        pk[i] = pack_bf16x2(e0, e1);
      }
      l = l * alpha + rs;
      m = m_new;

      if (j > 0) {
        // PV_{j-1} must be done: it reads the P tile and accumulates into O
        if (!wwait(&bars->o_done, (j - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            const uint32_t addr = tmem + lane_base + C::O_COL + cc * 32;
            tmem_ld32(addr, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(addr, o);
          }
          tmem_st_wait();
        }
      }
      // P row -> swizzled K-major tile: 16-byte piece q of chunk (keys 64*ch ..) at (q ^ (r % 8))
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int ch = q >> 3, qi = q & 7;
        uint4 v = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        *reinterpret_cast<uint4*>(prow + ch * C::CHUNK_BYTES + ((qi ^ rsw) << 4)) = v;
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }

    // ---- epilogue: O / l -> bf16, lse = ln2 * (m + log2 l)
    if (ok && nj > 0) {
      if (!wwait(&bars->o_done, (nj - 1) & 1)) ok = false;
      tc_fence_after();
    }
    if (!ok) fail(SITE_PF_SOFTMAX);
    const int h = kvh * p.g + h_local;
    const size_t row_index = (static_cast<size_t>(b) * p.Hq + h) * p.T + pos;
    __nv_bfloat16* orow = p.o + row_index * D;
    if (ok) {
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        if (nj > 0) {
          tmem_ld32(tmem + lane_base + C::O_COL + cc * 32, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (row_valid) {
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
      if (row_valid && p.lse) p.lse[row_index] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
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

int launch_prefill_tc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                      int T, int S, int d, float scale, int causal, cudaStream_t stream, unsigned* err,
                      unsigned long long timeout_ns) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return FA_ERR_CUDA;
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
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)B * Hkv};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)S * d * 2};
    cuuint32_t box[3] = {64, 128, 1};
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
  p.S = S;
  p.g = g;
  p.rows_per_head = rows_per_head;
  p.n_qtiles = (T + rows_per_head - 1) / rows_per_head;
  p.causal = causal;
  p.c = scale * kLog2e;
  p.err = err;
  p.timeout_ns = timeout_ns;
  const long long grid = static_cast<long long>(p.n_qtiles) * B * Hkv;
  if (grid > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (d == 128) {
    auto kfn = prefill_tc_kernel<128>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, PfCfg<128>::SMEM) != cudaSuccess)
      return FA_ERR_CUDA;
    kfn<<<static_cast<unsigned>(grid), PfCfg<128>::THREADS, PfCfg<128>::SMEM, stream>>>(tq, tk, tv, p);
  } else {
    auto kfn = prefill_tc_kernel<64>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, PfCfg<64>::SMEM) != cudaSuccess)
      return FA_ERR_CUDA;
    kfn<<<static_cast<unsigned>(grid), PfCfg<64>::THREADS, PfCfg<64>::SMEM, stream>>>(tq, tk, tv, p);
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
