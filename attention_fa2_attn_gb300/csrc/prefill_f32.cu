// prefill_f32.cu -- the same forward in FP32 throughout, on the CUDA cores.
//
// For problems that must match the fp64 oracle to 1e-5 (tensor-core tf32
// cannot). Same recurrence as the tensor-core kernel ("Kernel visualization:
// Flash Attention 1", "The tiled version"; FlashAttention-2 order with the
// division by l after the last tile), but with expf/logf and fp32 operands.
//
// One CTA = 32 query rows of one (batch, head); 128 threads. Per 32-key tile:
//   scores  -- thread (row = t % 32, key group = t / 32) computes 8 scores;
//   softmax -- warp w owns rows 8w..8w+7, one key per lane, shuffles for the
//              row max and sum;
//   P V     -- thread (row = t % 32, columns t/32 + 4i) accumulates O in
//              registers, rescaled by exp(m_old - m_new) per row.
#include "common.cuh"

namespace fa {

constexpr int F32_BR = 32;
constexpr int F32_BC = 32;
constexpr int F32_DMAX = 128;

struct F32Params {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  int B, Hq, Hkv, T, S, d, causal;
  float scale;
};

__global__ void __launch_bounds__(128) prefill_f32_kernel(const F32Params p) {
  extern __shared__ float fsm[];
  const int dp = p.d + 1;  // padded row pitch for the row-indexed tiles
  float* sQ = fsm;                      // [BR][d+1]
  float* sK = sQ + F32_BR * dp;         // [BC][d]   (read with the key uniform across a warp)
  float* sV = sK + F32_BC * p.d;        // [BC][d]
  float* sP = sV + F32_BC * p.d;        // [BR][BC+1]
  float* sAlpha = sP + F32_BR * (F32_BC + 1);  // [BR]

  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int bh = blockIdx.y;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int kvh = h / (p.Hq / p.Hkv);
  const int r0 = blockIdx.x * F32_BR;
  const float* qp = p.q + (static_cast<size_t>(b) * p.Hq + h) * p.T * p.d;
  const float* kp = p.k + (static_cast<size_t>(b) * p.Hkv + kvh) * p.S * p.d;
  const float* vp = p.v + (static_cast<size_t>(b) * p.Hkv + kvh) * p.S * p.d;
  const int shift = p.S - p.T;

  for (int x = t; x < F32_BR * p.d; x += 128) {
    const int r = x / p.d, c = x % p.d;
    sQ[r * dp + c] = (r0 + r < p.T) ? qp[static_cast<size_t>(r0 + r) * p.d + c] : 0.f;
  }
  // key range this row block can see
  int kv_end = p.S;
  if (p.causal) kv_end = max(0, min(p.S, min(r0 + F32_BR, p.T) - 1 + shift + 1));

  float m_row = -INFINITY, l_row = 0.f;  // carried by lane (row 8*warp + lane) for lane < 8
  const int orow = t & 31;
  const int ocol0 = t >> 5;
  float acc[F32_DMAX / 4];
#pragma unroll
  for (int i = 0; i < F32_DMAX / 4; ++i) acc[i] = 0.f;

  for (int k0 = 0; k0 < kv_end; k0 += F32_BC) {
    __syncthreads();
    for (int x = t; x < F32_BC * p.d; x += 128) {
      const int r = x / p.d, c = x % p.d;
      const bool in = k0 + r < p.S;
      sK[x] = in ? kp[static_cast<size_t>(k0 + r) * p.d + c] : 0.f;
      sV[x] = in ? vp[static_cast<size_t>(k0 + r) * p.d + c] : 0.f;
    }
    __syncthreads();
    {  // scores
      const int r = t & 31;
      const int kg = t >> 5;
      for (int kk = 0; kk < 8; ++kk) {
        const int key = kg * 8 + kk;
        float s = 0.f;
        for (int c = 0; c < p.d; ++c) s = fmaf(sQ[r * dp + c], sK[key * p.d + c], s);
        s *= p.scale;
        const int kj = k0 + key;
        const int qi = r0 + r;
        if (kj >= p.S || (p.causal && kj > qi + shift)) s = -INFINITY;
        sP[r * (F32_BC + 1) + key] = s;
      }
    }
    __syncthreads();
    // online softmax: warp w owns rows 8w..8w+7; lane = key
    for (int rr = 0; rr < 8; ++rr) {
      const int r = warp * 8 + rr;
      const float s = sP[r * (F32_BC + 1) + lane];
      float mx = s;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_old = __shfl_sync(0xffffffffu, m_row, rr);
      const float l_old = __shfl_sync(0xffffffffu, l_row, rr);
      const float m_new = fmaxf(m_old, mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float e = expf(s - m_use);
      float sum = e;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      const float alpha = expf(m_old - m_use);
      sP[r * (F32_BC + 1) + lane] = e;
      if (lane == rr) {
        m_row = m_new;
        l_row = l_old * alpha + sum;
      }
      if (lane == 0) sAlpha[r] = alpha;
    }
    __syncthreads();
    {  // O = alpha * O + P V
      const float a = sAlpha[orow];
      for (int i = 0; i < F32_DMAX / 4; ++i) {
        const int c = ocol0 + 4 * i;
        if (c >= p.d) break;
        float x = acc[i] * a;
        for (int key = 0; key < F32_BC; ++key) x = fmaf(sP[orow * (F32_BC + 1) + key], sV[key * p.d + c], x);
        acc[i] = x;
      }
    }
  }
  __syncthreads();
  // publish the final (m, l) of every row
  if (lane < 8) {
    sAlpha[warp * 8 + lane] = l_row;
    sP[warp * 8 + lane] = m_row;  // the score tile is free now
  }
  __syncthreads();
  const int qi = r0 + orow;
  if (qi < p.T) {
    const float l = sAlpha[orow];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* op = p.o + ((static_cast<size_t>(b) * p.Hq + h) * p.T + qi) * p.d;
    for (int i = 0; i < F32_DMAX / 4; ++i) {
      const int c = ocol0 + 4 * i;
      if (c >= p.d) break;
      op[c] = acc[i] * inv;
    }
    if (p.lse && ocol0 == 0)
      p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.T + qi] = l > 0.f ? sP[orow] + logf(l) : -INFINITY;
  }
}

int launch_prefill_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int Hq, int Hkv,
                       int T, int S, int d, float scale, int causal, cudaStream_t stream) {
  F32Params p{q, k, v, o, lse, B, Hq, Hkv, T, S, d, causal, scale};
  const size_t smem =
      sizeof(float) * (F32_BR * (d + 1) + 2 * F32_BC * d + F32_BR * (F32_BC + 1) + F32_BR);
  if (cudaFuncSetAttribute(prefill_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return FA_ERR_CUDA;
  dim3 grid((T + F32_BR - 1) / F32_BR, B * Hq);
  if (grid.y > 65535u) return FA_ERR_UNSUPPORTED;
  prefill_f32_kernel<<<grid, 128, smem, stream>>>(p);
  return launch_status();
}

}  // namespace fa
