// decode.cu -- split-KV decode (contiguous or paged K/V) and the log-sum-exp merge.
//
// What it computes:
//   * each CTA owns one key range ("split") of one (batch, KV head) and the
//     g*T query rows of that head's group stacked as one 16-row tile ("GQA
//     loads KV once per group"); it writes the normalised partial output of
//     its range and the range's lse ("Attention kernel chains", "The
//     log-sum-exp merge"), or the final bf16 O and lse when there is one
//     split. Key ranges are contiguous, c = ceil(S / n) rounded up to a
//     multiple of 64 keys.
//   * query row i of T sits at position S - T + i and sees key j iff
//     j <= i + (S - T) ("The causal mask for a decode step").
//   * paged: token t of sequence b is slot t % 16 of pool page
//     block_table[b][t / 16] ("The block-table cost of paged attention").
//   * merge: lse = ln sum_s e^{lse_s}, O = sum_s e^{lse_s - lse} O_s.
//
// How (GB300-specific): decode reads every K/V byte once and does 2*g FLOP
// per byte, so it is bound by HBM bandwidth. One producer warp streams
// 64-key K and V tiles with TMA (128-byte swizzle) into a shared-memory ring
// (4 stages of 32 KB, one CTA per SM, for contiguous K/V; 3 stages, two CTAs
// per SM, for paged K/V) -- 128 KB or more in flight per SM -- and the four consumer warps each
// take 16 keys of every tile. The 16 x 16 score block and the 16 x d output
// update of a warp are warp-level bf16 MMAs (m16n8k16), so the ALUs stay far
// from being a second bound; each warp keeps its own running max / sum /
// output and the four are merged through shared memory at the end. For paged
// K/V, the producer warp fetches 32 block-table entries at a time (one per
// lane) one batch ahead, and issues one TMA box per 16-token page.
#include "common.cuh"

namespace fa {

template <int D, int STAGES>
struct DecCfg {
  static constexpr int BC = 64;           // keys per tile
  static constexpr int KCH = D / 64;      // 128-byte chunks along d
  static constexpr int CHUNK = BC * 128;  // 64 rows x 128 bytes
  static constexpr int TILE = BC * D * 2; // bytes of one K (or V) tile
  static constexpr int STAGE_BYTES = 2 * TILE;
  static constexpr int OFF_BAR = STAGES * STAGE_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr int THREADS = 160;     // 4 consumer warps + 1 producer warp
};

struct DecParams {
  const __nv_bfloat16* q;
  __nv_bfloat16* o;  // final output (num_splits == 1)
  float* lse;        // final lse, may be null (num_splits == 1)
  float* o_part;     // [n][rows_total][D] (num_splits > 1)
  float* lse_part;   // [n][rows_total]
  const int* block_table;
  const int* seqlens;
  int B, Hq, Hkv, T, S;
  int g, rows;  // rows = g * T <= 16
  int num_splits;
  int max_pages, num_pages;
  int causal;
  float c;  // scale * log2(e)
  unsigned* err;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// byte offset of (row, d) inside a tile stored as KCH chunks of [64 rows][128 B], 128-byte swizzle
__device__ __forceinline__ uint32_t sw_off(int row, int d, int chunk_bytes) {
  const int ch = d >> 6;
  const int piece = (d & 63) >> 3;
  return ch * chunk_bytes + row * 128 + ((piece ^ (row & 7)) << 4) + ((d & 7) << 1);
}

// Paged decode runs two CTAs per SM (3-stage ring, 96 KB each): with 16-token
// pages a sequence is many small boxes, and two independent streams per SM keep
// more of them in flight. Contiguous split-KV runs one CTA per SM (4 stages).
template <int D, int STAGES, bool PAGED>
__global__ void __launch_bounds__(160, PAGED ? 2 : 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecParams p) {
  using C = DecCfg<D, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STAGES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv;
  const int kvh = bh % p.Hkv;

  // launched as a programmatic dependent of the previous launch on the stream (for a
  // decode loop, the previous step's merge, which still reads the partials this grid
  // overwrites): nothing global is read or written before that launch has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int S_b = p.S;
  if (PAGED) S_b = max(0, min(p.seqlens[b], p.max_pages * 16));
  const int per = (S_b + p.num_splits - 1) / p.num_splits;
  const int chunk = ((per + C::BC - 1) / C::BC) * C::BC;
  const int k_begin = min(S_b, split * chunk);
  const int k_end = min(S_b, k_begin + chunk);
  const int ntiles = (k_end - k_begin + C::BC - 1) / C::BC;
  const int shift = S_b - p.T;
  const uint64_t tmo = p.timeout_ns;
  const uint64_t tmo_unwind = unwind_timeout(tmo);  // copies landing before exit

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 4) {
    // ======================= producer warp =======================
    const int* trow = PAGED ? p.block_table + static_cast<size_t>(b) * p.max_pages : nullptr;
    const int first_page = k_begin >> 4;
    const int n_pages = (k_end - k_begin + 15) >> 4;  // pages holding keys of this range
    auto table_batch = [&](int bi) -> int {
      const int pg = bi * 32 + lane;
      return (PAGED && pg < n_pages) ? __ldg(trow + first_page + pg) : -1;
    };
    int cur = 0, nxt = 0, cur_batch = -1;
    if (PAGED && ntiles > 0) {
      nxt = table_batch(0);
    }
    int issued = 0;
    bool ok = true;
    for (int it = 0; it < ntiles; ++it) {
      const int s = it % STAGES;
      const uint32_t u = it / STAGES;
      if (PAGED) {
        const int batch = it >> 3;  // 8 tiles of 4 pages per 32-entry batch
        if (batch != cur_batch) {
          cur = nxt;
          nxt = table_batch(batch + 1);
          cur_batch = batch;
        }
      }
      bool w = true;
      if (it >= STAGES) w = mbar_wait(&empty[s], (u - 1) & 1, tmo, abort_flag);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      uint8_t* sK = smem + s * C::STAGE_BYTES;
      uint8_t* sV = sK + C::TILE;
      const int key0 = k_begin + it * C::BC;
      if (!PAGED) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          for (int c = 0; c < C::KCH; ++c) {
            tma_load_3d(sK + c * C::CHUNK, &tmK, &full[s], c * 64, key0, bh);
            tma_load_3d(sV + c * C::CHUNK, &tmV, &full[s], c * 64, key0, bh);
          }
        }
      } else {
        int ent[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ent[i] = __shfl_sync(0xffffffffu, cur, (it & 7) * 4 + i);
        if (lane == 0) {
          int pages_ok = 0;
          bool loads[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const bool in_range = (it * 4 + i) < n_pages;
            const bool valid = ent[i] >= 0 && ent[i] < p.num_pages;
            if (in_range && !valid) record_error(p.err, FA_ERR_BOUNDS, SITE_DEC_TABLE);
            loads[i] = in_range && valid;
            pages_ok += loads[i] ? 1 : 0;
          }
          // bytes actually requested: one K and one V box per loaded page and d-chunk
          mbar_arrive_expect_tx(&full[s], pages_ok * 2 * C::KCH * 16 * 128);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (!loads[i]) continue;
            for (int c = 0; c < C::KCH; ++c) {
              tma_load_3d(sK + c * C::CHUNK + i * 16 * 128, &tmK, &full[s], c * 64, kvh, ent[i] * 16);
              tma_load_3d(sV + c * C::CHUNK + i * 16 * 128, &tmV, &full[s], c * 64, kvh, ent[i] * 16);
            }
          }
        }
      }
      issued = it + 1;
    }
    if (!ok) {
      if (lane == 0) {
        record_error(p.err, FA_ERR_TIMEOUT, SITE_DEC_PRODUCER);
        *abort_flag = 1;
        for (int it = max(0, issued - STAGES); it < issued; ++it)
          mbar_wait(&full[it % STAGES], (it / STAGES) & 1, tmo_unwind);
      }
    }
  } else {
    // ======================= consumer warps 0-3 =======================
    const int gid = lane >> 2;  // row of the MMA fragment (and +8)
    const int tig = lane & 3;
    // Q fragments (A operand, rows = stacked (head, position) pairs)
    uint32_t qa[D / 16][4];
    {
      const uint32_t* qrow[2] = {nullptr, nullptr};
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        const int r = gid + 8 * ri;
        if (r < p.rows) {
          const int h = kvh * p.g + r / p.T;
          const int t = r % p.T;
          qrow[ri] = reinterpret_cast<const uint32_t*>(p.q + ((static_cast<size_t>(b) * p.Hq + h) * p.T + t) * D);
        }
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        qa[kk][0] = qrow[0] ? __ldg(qrow[0] + kk * 8 + tig) : 0u;
        qa[kk][1] = qrow[1] ? __ldg(qrow[1] + kk * 8 + tig) : 0u;
        qa[kk][2] = qrow[0] ? __ldg(qrow[0] + kk * 8 + 4 + tig) : 0u;
        qa[kk][3] = qrow[1] ? __ldg(qrow[1] + kk * 8 + 4 + tig) : 0u;
      }
    }
    // visibility limit of the two rows this thread holds
    int lim[2];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      const int r = gid + 8 * ri;
      const int t = (r < p.rows) ? r % p.T : 0;
      lim[ri] = p.causal ? min(k_end - 1, t + shift) : k_end - 1;
    }
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    const float c = p.c;
    bool ok = true;

    for (int it = 0; it < ntiles; ++it) {
      const int s = it % STAGES;
      const bool w = mbar_wait(&full[s], (it / STAGES) & 1, tmo, abort_flag);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      uint8_t* sK = smem + s * C::STAGE_BYTES;
      uint8_t* sV = sK + C::TILE;
      const uint32_t sKa = smem_u32(sK), sVa = smem_u32(sV);
      const int key0 = k_begin + it * C::BC;
      const int wrow0 = warp * 16;  // this warp's first key row in the tile

      // ---- S = Q K^T for this warp's 16 keys
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int mi = lane >> 3;  // matrix index 0..3 = (n-tile, d half)
        const int row = wrow0 + 8 * (mi >> 1) + (lane & 7);
        const int dcol = kk * 16 + 8 * (mi & 1);
        uint32_t b00, b01, b10, b11;
        ldsm_x4(sKa + sw_off(row, dcol, C::CHUNK), b00, b01, b10, b11);
        mma_bf16_16816(acc[0], qa[kk], b00, b01);
        mma_bf16_16816(acc[1], qa[kk], b10, b11);
      }
      // ---- mask: keys past the range end or (causal) after the row's position
      const bool tail = key0 + C::BC > k_end;
      if (tail || p.causal) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = key0 + wrow0 + 8 * nt + 2 * tig + (e & 1);
            if (key > lim[e >> 1]) acc[nt][e] = -INFINITY;
          }
      }
      // ---- online softmax (two rows per thread; a quad of threads shares a row)
      float alpha[2];
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        float mx = fmaxf(fmaxf(acc[0][2 * ri], acc[0][2 * ri + 1]), fmaxf(acc[1][2 * ri], acc[1][2 * ri + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m[ri], mx * c);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        alpha[ri] = ex2_approx(m[ri] - m_use);
        float sum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pv = ex2_approx(fmaf(acc[nt][2 * ri + e], c, -m_use));
            acc[nt][2 * ri + e] = pv;
            sum += pv;
          }
        l[ri] = l[ri] * alpha[ri] + sum;
        m[ri] = m_new;
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
      uint32_t pa[4];
      pa[0] = pack_bf16x2(acc[0][0], acc[0][1]);
      pa[1] = pack_bf16x2(acc[0][2], acc[0][3]);
      pa[2] = pack_bf16x2(acc[1][0], acc[1][1]);
      pa[3] = pack_bf16x2(acc[1][2], acc[1][3]);
      // ---- keys past the range end: zero this warp's V rows so stale or
      //      unloaded bytes cannot reach O through a zero weight (0 * NaN)
      if (tail) {
        for (int idx = lane; idx < 16 * (D / 8); idx += 32) {
          const int rr = idx / (D / 8);
          const int dd = (idx % (D / 8)) * 8;
          if (key0 + wrow0 + rr >= k_end)
            *reinterpret_cast<uint4*>(sV + sw_off(wrow0 + rr, dd, C::CHUNK)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_async_smem();  // order these generic writes before the next TMA write to the stage
        __syncwarp();
      }
      // ---- O += P V (B operand = V rows of this warp's keys, transposed load)
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        const int mi = lane >> 3;  // (keys half, d half)
        const int row = wrow0 + 8 * (mi & 1) + (lane & 7);
        const int dcol = np * 16 + 8 * (mi >> 1);
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(sVa + sw_off(row, dcol, C::CHUNK), v0, v1, v2, v3);
        mma_bf16_16816(o[2 * np], pa, v0, v1);
        mma_bf16_16816(o[2 * np + 1], pa, v2, v3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!ok) {
      if (lane == 0) {
        record_error(p.err, FA_ERR_TIMEOUT, SITE_DEC_CONSUMER);
        *abort_flag = 1;
      }
    }

    // the LSE merge of the split partials (a dependent launch) may be scheduled now;
    // it still waits for this grid to finish before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // ---- merge the four warps' (m, l, O) through shared memory
    float lt[2];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      float x = l[ri];
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      lt[ri] = x;
    }
    named_bar_sync(1, 128);  // every consumer is past its last tile: the ring is free
    float* wO = reinterpret_cast<float*>(smem);       // [4 warps][16 rows][D]
    float* wM = wO + 4 * 16 * D;                      // [4][16]
    float* wL = wM + 4 * 16;                          // [4][16]
    if (!*abort_flag) {
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        const int col = n * 8 + 2 * tig;
        wO[(warp * 16 + gid) * D + col] = o[n][0];
        wO[(warp * 16 + gid) * D + col + 1] = o[n][1];
        wO[(warp * 16 + gid + 8) * D + col] = o[n][2];
        wO[(warp * 16 + gid + 8) * D + col + 1] = o[n][3];
      }
      if (tig == 0) {
        wM[warp * 16 + gid] = m[0];
        wM[warp * 16 + gid + 8] = m[1];
        wL[warp * 16 + gid] = lt[0];
        wL[warp * 16 + gid + 8] = lt[1];
      }
    }
    named_bar_sync(1, 128);
    if (!*abort_flag) {
      const int t = threadIdx.x;  // 0..127
      const int r = t >> 3;       // row 0..15
      const int c0 = (t & 7) * (D / 8);
      if (r < p.rows) {
        float M = -INFINITY;
        for (int w = 0; w < 4; ++w) M = fmaxf(M, wM[w * 16 + r]);
        float scl[4];
        float L = 0.f;
        for (int w = 0; w < 4; ++w) {
          scl[w] = (M == -INFINITY) ? 0.f : ex2_approx(wM[w * 16 + r] - M);
          L += wL[w * 16 + r] * scl[w];
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const int h = kvh * p.g + r / p.T;
        const size_t row_g = (static_cast<size_t>(b) * p.Hq + h) * p.T + (r % p.T);
        const float lse_v = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        if (p.num_splits == 1) {
          __nv_bfloat16* dst = p.o + row_g * D + c0;
          for (int cc = 0; cc < D / 8; cc += 2) {
            float a0 = 0.f, a1 = 0.f;
            for (int w = 0; w < 4; ++w) {
              a0 += wO[(w * 16 + r) * D + c0 + cc] * scl[w];
              a1 += wO[(w * 16 + r) * D + c0 + cc + 1] * scl[w];
            }
            *reinterpret_cast<uint32_t*>(dst + cc) = pack_bf16x2(a0 * inv, a1 * inv);
          }
          if (p.lse && (t & 7) == 0) p.lse[row_g] = lse_v;
        } else {
          const size_t rows_total = static_cast<size_t>(p.B) * p.Hq * p.T;
          float* dst = p.o_part + (static_cast<size_t>(split) * rows_total + row_g) * D + c0;
          for (int cc = 0; cc < D / 8; ++cc) {
            float a = 0.f;
            for (int w = 0; w < 4; ++w) a += wO[(w * 16 + r) * D + c0 + cc] * scl[w];
            dst[cc] = a * inv;
          }
          if ((t & 7) == 0) p.lse_part[static_cast<size_t>(split) * rows_total + row_g] = lse_v;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// LSE merge: one warp per output row
// ---------------------------------------------------------------------------
// lse = ln sum_s e^{lse_s};  O = sum_s e^{lse_s - lse} O_s. Lane s reads split s's
// lse once (32 splits at a time) and the row's max, sum and weights come from warp
// shuffles; the weight of split s is then broadcast from its lane while every lane
// reads its NJ columns (col = lane + 32 j) of O_s. A row costs one round trip for
// the lse values and one per G splits for the partials.
template <int NJ, int G>
__global__ void __launch_bounds__(128) lse_merge_kernel(const float* __restrict__ o_part,
                                                        const float* __restrict__ lse_part,
                                                        __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                        int n, int rows, int d) {
  // launched as a programmatic dependent of the split kernel: wait until that grid
  // has finished and its partials are visible (a no-op for a plain launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next launch on the stream may start now; it waits for this grid before it
  // touches anything (the next decode step overwrites the partials read here)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const size_t step = static_cast<size_t>(rows) * d;  // one split's partials
  const float ls0 = lane < n ? lse_part[static_cast<size_t>(lane) * rows + row] : -INFINITY;
  float mx = ls0;
  for (int s = 32 + lane; s < n; s += 32) mx = fmaxf(mx, lse_part[static_cast<size_t>(s) * rows + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float tot = 0.f;
  if (mx != -INFINITY) {
    if (ls0 != -INFINITY) tot = expf(ls0 - mx);
    for (int s = 32 + lane; s < n; s += 32) {
      const float ls = lse_part[static_cast<size_t>(s) * rows + row];
      if (ls != -INFINITY) tot += expf(ls - mx);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
  const float lrow = (mx == -INFINITY) ? -INFINITY : mx + logf(tot);
  float acc[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) acc[j] = 0.f;
  if (mx != -INFINITY) {
    for (int s0 = 0; s0 < n; s0 += 32) {
      // weight of split s0 + lane; 0 for an empty split (its O_s is never read)
      const float ls = s0 == 0 ? ls0 : (s0 + lane < n ? lse_part[static_cast<size_t>(s0 + lane) * rows + row] : -INFINITY);
      const float ws = ls != -INFINITY ? expf(ls - lrow) : 0.f;
      const int cnt = min(32, n - s0);
      const float* src = o_part + (static_cast<size_t>(s0) * rows + row) * d + lane;
      // G splits' partials are loaded before any is used, so their loads overlap; an
      // empty split's partial is read (it lies inside the buffer) but gets no weight
      for (int g0 = 0; g0 < cnt; g0 += G) {
        float v[G][NJ];
#pragma unroll
        for (int i = 0; i < G; ++i)
#pragma unroll
          for (int j = 0; j < NJ; ++j)
            v[i][j] = (g0 + i < cnt && lane + 32 * j < d) ? src[(g0 + i) * step + 32 * j] : 0.f;
#pragma unroll
        for (int i = 0; i < G; ++i) {
          const float w = __shfl_sync(0xffffffffu, ws, (g0 + i) & 31);
          if (g0 + i < cnt && w != 0.f) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) acc[j] = fmaf(w, v[i][j], acc[j]);
          }
        }
      }
    }
  }
  __nv_bfloat16* dst = o + static_cast<size_t>(row) * d + lane;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    if (lane + 32 * j < d) dst[32 * j] = __float2bfloat16_rn(acc[j]);
  if (lse && lane == 0) lse[row] = lrow;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();

template <bool PAGED>
constexpr int dec_stages() { return PAGED ? 3 : 4; }

// `after_split`: launched right behind the kernel that wrote the partials, on the
// same stream, as a programmatic dependent (its launch overlaps that kernel's tail;
// griddepcontrol.wait holds it until the partials are complete and visible).
static int launch_lse_merge_impl(const float* o_part, const float* lse_part, void* o, float* lse, int n, int rows,
                                 int d, cudaStream_t stream, bool after_split) {
  if (d < 1 || d > 256) return FA_ERR_UNSUPPORTED;
  const int grid = static_cast<int>((static_cast<long long>(rows) + 3) / 4);  // one warp per row
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_split ? 1 : 0;
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
  // loads in flight per lane: G splits x NJ columns. Many splits (decode) take the wider
  // group; a few (the prefill key split, thousands of rows) the narrower one, which
  // keeps more warps resident.
  const bool wide = n >= 12;
  cudaError_t e;
  if (d <= 32)
    e = wide ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<1, 8>, o_part, lse_part, ob, lse, n, rows, d)
             : cudaLaunchKernelEx(&cfg, lse_merge_kernel<1, 4>, o_part, lse_part, ob, lse, n, rows, d);
  else if (d <= 64)
    e = wide ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<2, 8>, o_part, lse_part, ob, lse, n, rows, d)
             : cudaLaunchKernelEx(&cfg, lse_merge_kernel<2, 4>, o_part, lse_part, ob, lse, n, rows, d);
  else if (d <= 128)
    e = wide ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<4, 8>, o_part, lse_part, ob, lse, n, rows, d)
             : cudaLaunchKernelEx(&cfg, lse_merge_kernel<4, 4>, o_part, lse_part, ob, lse, n, rows, d);
  else
    e = wide ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<8, 4>, o_part, lse_part, ob, lse, n, rows, d)
             : cudaLaunchKernelEx(&cfg, lse_merge_kernel<8, 2>, o_part, lse_part, ob, lse, n, rows, d);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  return launch_status();
}

int launch_lse_merge(const float* o_part, const float* lse_part, void* o, float* lse, int n, int rows, int d,
                     cudaStream_t stream, bool after_split) {
  return launch_lse_merge_impl(o_part, lse_part, o, lse, n, rows, d, stream, after_split);
}

template <int D, bool PAGED>
static int launch_decode_t(const CUtensorMap& tk, const CUtensorMap& tv, const DecParams& p, int nsplit, int nbh,
                           cudaStream_t stream) {
  constexpr int ST = dec_stages<PAGED>();
  using C = DecCfg<D, ST>;
  auto kfn = decode_kernel<D, ST, PAGED>;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  // a programmatic dependent of the previous launch on the stream: the launch and the
  // CTAs' start overlap that launch's tail; the kernel waits before any global access
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nsplit, nbh);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kfn, tk, tv, p) != cudaSuccess) return FA_ERR_CUDA;
  return launch_status();
}

// Shared by the contiguous and the paged entry points. `k`/`v` are either
// [B][Hkv][S][d] (contiguous) or pools [num_pages][16][Hkv][d] (paged).
int launch_decode(const void* q, const void* k, const void* v, const int* block_table, const int* seqlens, void* o,
                  float* lse, int B, int Hq, int Hkv, int T, int S, int max_pages, int num_pages, int d, float scale,
                  int causal, int num_splits, void* workspace, cudaStream_t stream, unsigned* err,
                  unsigned long long timeout_ns) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return FA_ERR_CUDA;
  const bool paged = block_table != nullptr;
  CUtensorMap tk, tv;
  for (int w = 0; w < 2; ++w) {
    cuuint64_t dims[3];
    cuuint64_t strides[2];
    cuuint32_t box[3];
    if (!paged) {
      dims[0] = d; dims[1] = S; dims[2] = static_cast<cuuint64_t>(B) * Hkv;
      strides[0] = static_cast<cuuint64_t>(d) * 2;
      strides[1] = static_cast<cuuint64_t>(S) * d * 2;
      box[0] = 64; box[1] = 64; box[2] = 1;
    } else {
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
  const size_t rows_total = static_cast<size_t>(B) * Hq * T;
  DecParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.o_part = nullptr;
  p.lse_part = nullptr;
  if (num_splits > 1) {
    p.o_part = static_cast<float*>(workspace);
    const size_t obytes = ((static_cast<size_t>(num_splits) * rows_total * d * 4 + 255) / 256) * 256;
    p.lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + obytes);
  }
  p.block_table = block_table;
  p.seqlens = seqlens;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.T = T;
  p.S = S;
  p.g = Hq / Hkv;
  p.rows = p.g * T;
  p.num_splits = num_splits;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.causal = causal;
  p.c = scale * kLog2e;
  p.err = err;
  p.timeout_ns = timeout_ns;
  const int nbh = B * Hkv;
  int rc;
  if (d == 128)
    rc = paged ? launch_decode_t<128, true>(tk, tv, p, num_splits, nbh, stream)
               : launch_decode_t<128, false>(tk, tv, p, num_splits, nbh, stream);
  else
    rc = paged ? launch_decode_t<64, true>(tk, tv, p, num_splits, nbh, stream)
               : launch_decode_t<64, false>(tk, tv, p, num_splits, nbh, stream);
  if (rc != FA_OK || num_splits == 1) return rc;
  return launch_lse_merge_impl(p.o_part, p.lse_part, o, lse, num_splits, static_cast<int>(rows_total), d, stream,
                               true);
}

}  // namespace fa
