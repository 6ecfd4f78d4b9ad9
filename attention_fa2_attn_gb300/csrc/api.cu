// api.cu -- the extern "C" boundary declared in include/fa_gb300.h:
// argument validation, the split-count heuristic, the device error word,
// tensor-map encoder lookup and kernel dispatch.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"

namespace fa {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int launch_prefill_tc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                      int T, int S, int d, float scale, int causal, cudaStream_t stream, unsigned* err,
                      unsigned long long timeout_ns, const int* block_table, const int* seqlens, int max_pages,
                      int num_pages, int num_splits, float* o_part, float* lse_part);
int launch_prefill_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int Hq, int Hkv,
                       int T, int S, int d, float scale, int causal, cudaStream_t stream);
int launch_decode(const void* q, const void* k, const void* v, const int* block_table, const int* seqlens, void* o,
                  float* lse, int B, int Hq, int Hkv, int T, int S, int max_pages, int num_pages, int d, float scale,
                  int causal, int num_splits, void* workspace, cudaStream_t stream, unsigned* err,
                  unsigned long long timeout_ns);
int launch_lse_merge(const float* o_part, const float* lse_part, void* o, float* lse, int n, int rows, int d,
                     cudaStream_t stream, bool after_split);
int launch_backward(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* d_o,
                    void* dq, void* dk, void* dv, float* vecs, int B, int Hq, int Hkv, int T, int S, int d,
                    float scale, int causal, cudaStream_t stream, unsigned* err, unsigned long long timeout_ns);
int launch_kv_outer(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int T,
                    int S, int d, float scale, int causal, int row_bands, void* workspace, cudaStream_t stream,
                    unsigned* err, unsigned long long timeout_ns);

// The device-side error word (code | site << 8). Kernels receive its device
// address as a parameter.
__device__ unsigned g_fa_device_error;

static thread_local char g_cuda_err[256] = "no error";
static unsigned long long g_timeout_ns = 4000000000ull;
// The settable wait bound never goes below this: a shorter one would report
// timeouts that are not faults whenever the GPU is time-sliced with other work.
static constexpr unsigned long long kMinWaitTimeoutNs = 1000000ull;  // 1 ms

// Keeps the text of a CUDA error for fa_last_cuda_error_string; cudaSuccess (the
// error was already consumed and recorded where it happened) keeps the old text.
static int cuda_fail(cudaError_t e) {
  if (e != cudaSuccess)
    snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return FA_ERR_CUDA;
}

static std::mutex g_mu;

EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !ptr) {
      cuda_fail(e != cudaSuccess ? e : cudaErrorSymbolNotFound);
      return nullptr;
    }
    fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Device address of the error word on the current device (looked up once per device).
static unsigned* error_word() {
  static unsigned* addr[128] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned*>(p);
  }
  return addr[dev];
}

static int sm_count() {
  static int cnt[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  if (!cnt[dev]) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cnt[dev] = c;
  }
  return cnt[dev];
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool good_scale(float s) { return isfinite(s) && s > 0.f; }

__global__ void selftest_wait_kernel(unsigned* err, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: the bounded wait must give up and report
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, timeout_ns)) record_error(err, FA_ERR_TIMEOUT, SITE_SELFTEST);
}

// Accessors for other translation units of the library.
unsigned* device_error_word() { return error_word(); }
unsigned long long wait_timeout_ns() { return g_timeout_ns; }
int device_sm_count() { return sm_count(); }
int record_cuda_failure(cudaError_t e) { return cuda_fail(e); }

}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 100; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_BOUNDS: return "FA_ERR_BOUNDS";
    default: return "FA_ERR_UNKNOWN";
  }
}

const char* fa_last_cuda_error_string(void) { return g_cuda_err; }

void fa_set_wait_timeout_ns(unsigned long long ns) { g_timeout_ns = ns < kMinWaitTimeoutNs ? kMinWaitTimeoutNs : ns; }

void fa_get_wait_timeouts(unsigned long long* wait_ns, unsigned long long* unwind_ns) {
  if (wait_ns) *wait_ns = g_timeout_ns;
  if (unwind_ns) *unwind_ns = unwind_timeout(g_timeout_ns);
}

int fa_num_splits_heuristic(int B, int Hkv, int S, int num_sms) {
  if (B <= 0 || Hkv <= 0 || S <= 0 || num_sms <= 0) return 1;
  const long long units = static_cast<long long>(B) * Hkv;
  if (units >= num_sms) return 1;
  long long n = num_sms / units;             // fill at most one wave
  const long long cap = (S + 255) / 256;     // at least 256 keys per split
  if (n > cap) n = cap;
  if (n > 1024) n = 1024;
  return n < 1 ? 1 : static_cast<int>(n);
}

int fa_num_splits_prefill(int B, int Hq, int Hkv, int T, int S, int num_sms) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || S <= 0 || num_sms <= 0 || Hq % Hkv != 0) return 1;
  const long long g = Hq / Hkv;
  if (g > 128) return 1;
  const long long rows_per_tile = 128 / g;                    // query positions per 128-row tile
  const long long tiles = (T + rows_per_tile - 1) / rows_per_tile;
  const long long units = (tiles + 1) / 2 * B * Hkv;          // query-tile pairs: the unsplit work items
  if (units >= num_sms) return 1;
  long long n = num_sms / units;                              // fill at most one wave
  const long long cap = (S + 511) / 512;                      // at least four 128-key tiles per range
  if (n > cap) n = cap;
  if (n > 64) n = 64;
  return n < 1 ? 1 : static_cast<int>(n);
}

// More than 16 stacked query rows per KV head (g * T > 16: chunked prefill or a
// multi-token decode step) go to the tensor-core prefill kernel, which tiles the
// queries itself; a key split is then only for shapes with too few query tiles to
// fill the GPU (contiguous K/V).
static bool many_rows(int Hq, int Hkv, int T) { return static_cast<long long>(Hq / Hkv) * T > 16; }

int fa_decode_num_splits(int B, int Hq, int Hkv, int T, int S, int paged, int num_sms) {
  if (B < 1 || Hq < 1 || Hkv < 1 || T < 1 || S < 1 || num_sms < 1 || Hq % Hkv != 0) return 1;
  if (many_rows(Hq, Hkv, T)) return paged ? 1 : fa_num_splits_prefill(B, Hq, Hkv, T, S, num_sms);
  return fa_num_splits_heuristic(B, Hkv, S, num_sms);
}

size_t fa_decode_workspace_bytes(int B, int Hq, int T, int d, int num_splits) {
  if (num_splits <= 1 || B <= 0 || Hq <= 0 || T <= 0 || d <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * T;
  const size_t obytes = ((static_cast<size_t>(num_splits) * rows * d * 4 + 255) / 256) * 256;
  return obytes + static_cast<size_t>(num_splits) * rows * 4;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Tq,
                 int Skv, int d, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Skv < 1 || Hq % Hkv != 0 || !good_scale(scale))
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const int g = Hq / Hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq * Tq >= (1ll << 31) || static_cast<long long>(B) * Hkv * Skv >= (1ll << 31))
    return FA_ERR_UNSUPPORTED;
  unsigned* err = error_word();
  if (!err) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
  int rc = launch_prefill_tc(q, k, v, o, lse, B, Hq, Hkv, Tq, Skv, d, scale, causal ? 1 : 0,
                             static_cast<cudaStream_t>(stream), err, g_timeout_ns, nullptr, nullptr, 0, 0, 1, nullptr,
                             nullptr);
  if (rc == FA_ERR_CUDA) cuda_fail(cudaGetLastError());
  return static_cast<fa_status>(rc);
}

size_t fa_bwd_workspace_bytes(int B, int Hq, int T) {
  if (B <= 0 || Hq <= 0 || T <= 0) return 0;
  const size_t t_pad = (static_cast<size_t>(T) + 3) / 4 * 4;
  return 2 * static_cast<size_t>(B) * Hq * t_pad * 4;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* d_o,
                 void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Tq, int Skv, int d, float scale, int causal,
                 void* workspace, size_t ws_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse || !d_o || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(d_o) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Skv < 1 || Hq % Hkv != 0 || !good_scale(scale))
    return FA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u) || ws_bytes < fa_bwd_workspace_bytes(B, Hq, Tq))
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const int g = Hq / Hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq * Tq >= (1ll << 31) || static_cast<long long>(B) * Hkv * Skv >= (1ll << 31))
    return FA_ERR_UNSUPPORTED;
  unsigned* err = error_word();
  if (!err) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
  int rc = launch_backward(q, k, v, o, lse, d_o, dq, dk, dv, static_cast<float*>(workspace), B, Hq, Hkv, Tq, Skv, d,
                           scale, causal ? 1 : 0, static_cast<cudaStream_t>(stream), err, g_timeout_ns);
  if (rc == FA_ERR_CUDA) cuda_fail(cudaGetLastError());
  return static_cast<fa_status>(rc);
}

size_t fa_fwd_kv_outer_workspace_bytes(int B, int Hq, int Tq, int d) {
  if (B <= 0 || Hq <= 0 || Tq <= 0 || d <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * Tq;
  return ((rows * d * 4 + 255) / 256) * 256 + 2 * rows * 4;
}

fa_status fa_fwd_kv_outer(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                          int Tq, int Skv, int d, float scale, int causal, int row_bands, void* workspace,
                          size_t ws_bytes, void* stream) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Skv < 1 || Hq % Hkv != 0 || !good_scale(scale) || row_bands < 1)
    return FA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || ws_bytes < fa_fwd_kv_outer_workspace_bytes(B, Hq, Tq, d))
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const int g = Hq / Hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq * Tq >= (1ll << 31) || static_cast<long long>(B) * Hkv * Skv >= (1ll << 31))
    return FA_ERR_UNSUPPORTED;
  unsigned* err = error_word();
  if (!err) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
  int rc = launch_kv_outer(q, k, v, o, lse, B, Hq, Hkv, Tq, Skv, d, scale, causal ? 1 : 0, row_bands, workspace,
                           static_cast<cudaStream_t>(stream), err, g_timeout_ns);
  if (rc == FA_ERR_CUDA) cuda_fail(cudaGetLastError());
  return static_cast<fa_status>(rc);
}

fa_status fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int Hq, int Hkv,
                     int Tq, int Skv, int d, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Skv < 1 || Hq % Hkv != 0 || !good_scale(scale))
    return FA_ERR_INVALID_ARG;
  if (d < 1 || d > 128) return FA_ERR_UNSUPPORTED;
  int rc = launch_prefill_f32(q, k, v, o, lse, B, Hq, Hkv, Tq, Skv, d, scale, causal ? 1 : 0,
                              static_cast<cudaStream_t>(stream));
  if (rc == FA_ERR_CUDA) cuda_fail(cudaGetLastError());
  return static_cast<fa_status>(rc);
}

static fa_status check_decode_common(const void* q, const void* o, int B, int Hq, int Hkv, int T, int d, float scale,
                                     int num_splits) {
  if (!q || !o) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || T < 1 || Hq % Hkv != 0 || !good_scale(scale)) return FA_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > 1024) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hkv > 65535) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq * T >= (1ll << 31)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

static fa_status check_many_rows(int Hq, int Hkv, int num_splits, bool paged) {
  const int g = Hq / Hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return FA_ERR_UNSUPPORTED;
  if (paged && num_splits > 1) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Splits that fit in ws_bytes (partials plus lse, as fa_decode_workspace_bytes lays them out).
static int splits_that_fit(int B, int Hq, int T, int d, int want, const void* workspace, size_t ws_bytes) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return 1;
  int n = want;
  while (n > 1 && fa_decode_workspace_bytes(B, Hq, T, d, n) > ws_bytes) --n;
  return n;
}

fa_status fa_decode_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                            int T, int S, int d, float scale, int causal, int num_splits, void* workspace,
                            size_t ws_bytes, void* stream) {
  fa_status st = check_decode_common(q, o, B, Hq, Hkv, T, d, scale, num_splits);
  if (st != FA_OK) return st;
  if (!k || !v || !aligned16(k) || !aligned16(v) || S < 1) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * Hkv * S >= (1ll << 31)) return FA_ERR_UNSUPPORTED;
  if (many_rows(Hq, Hkv, T)) {
    st = check_many_rows(Hq, Hkv, num_splits, false);
    if (st != FA_OK) return st;
    int n = num_splits;
    if (n == 0) {
      // heuristic, limited to what the given workspace holds (none: no split)
      const int sms = sm_count();
      if (!sms) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
      n = splits_that_fit(B, Hq, T, d, fa_decode_num_splits(B, Hq, Hkv, T, S, 0, sms), workspace, ws_bytes);
    } else if (n > 1) {
      if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID_ARG;
      if (ws_bytes < fa_decode_workspace_bytes(B, Hq, T, d, n)) return FA_ERR_INVALID_ARG;
    }
    unsigned* err = error_word();
    if (!err) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
    float* o_part = nullptr;
    float* lse_part = nullptr;
    const size_t rows = static_cast<size_t>(B) * Hq * T;
    if (n > 1) {
      o_part = static_cast<float*>(workspace);
      const size_t obytes = ((static_cast<size_t>(n) * rows * d * 4 + 255) / 256) * 256;
      lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + obytes);
    }
    int rc = launch_prefill_tc(q, k, v, o, lse, B, Hq, Hkv, T, S, d, scale, causal ? 1 : 0,
                               static_cast<cudaStream_t>(stream), err, g_timeout_ns, nullptr, nullptr, 0, 0, n, o_part,
                               lse_part);
    if (rc == FA_OK && n > 1)
      rc = launch_lse_merge(o_part, lse_part, o, lse, n, static_cast<int>(rows), d, static_cast<cudaStream_t>(stream),
                            true);
    if (rc == FA_ERR_CUDA) cuda_fail(cudaGetLastError());
    return static_cast<fa_status>(rc);
  }
  int n = num_splits;
  if (n == 0) {
    const int sms = sm_count();
    if (!sms) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
    n = fa_decode_num_splits(B, Hq, Hkv, T, S, 0, sms);
  }
  if (n > 1) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID_ARG;
    if (ws_bytes < fa_decode_workspace_bytes(B, Hq, T, d, n)) return FA_ERR_INVALID_ARG;
  }
  unsigned* err = error_word();
  if (!err) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
  int rc = launch_decode(q, k, v, nullptr, nullptr, o, lse, B, Hq, Hkv, T, S, 0, 0, d, scale, causal ? 1 : 0, n,
                         workspace, static_cast<cudaStream_t>(stream), err, g_timeout_ns);
  if (rc == FA_ERR_CUDA) cuda_fail(cudaGetLastError());
  return static_cast<fa_status>(rc);
}

fa_status fa_lse_merge(const float* o_part, const float* lse_part, void* o, float* lse, int num_splits, int rows,
                       int d, void* stream) {
  if (!o_part || !lse_part || !o) return FA_ERR_INVALID_ARG;
  if (num_splits < 1 || rows < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (d > 256) return FA_ERR_UNSUPPORTED;
  int rc = launch_lse_merge(o_part, lse_part, o, lse, num_splits, rows, d, static_cast<cudaStream_t>(stream), false);
  if (rc == FA_ERR_CUDA) cuda_fail(cudaGetLastError());
  return static_cast<fa_status>(rc);
}

fa_status fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                          const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv, int T, int max_pages,
                          int page_size, int num_pages, int d, float scale, int causal, int num_splits,
                          void* workspace, size_t ws_bytes, void* stream) {
  fa_status st = check_decode_common(q, o, B, Hq, Hkv, T, d, scale, num_splits);
  if (st != FA_OK) return st;
  if (!k_pages || !v_pages || !block_table || !seqlens) return FA_ERR_INVALID_ARG;
  if (!aligned16(k_pages) || !aligned16(v_pages) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seqlens) & 3u))
    return FA_ERR_INVALID_ARG;
  if (max_pages < 1 || num_pages < 1) return FA_ERR_INVALID_ARG;
  if (page_size != 16) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_pages) * 16 >= (1ll << 31) || static_cast<long long>(max_pages) * 16 >= (1ll << 31))
    return FA_ERR_UNSUPPORTED;
  if (many_rows(Hq, Hkv, T)) {
    st = check_many_rows(Hq, Hkv, num_splits, true);
    if (st != FA_OK) return st;
    unsigned* err = error_word();
    if (!err) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
    int rc = launch_prefill_tc(q, k_pages, v_pages, o, lse, B, Hq, Hkv, T, 0, d, scale, causal ? 1 : 0,
                               static_cast<cudaStream_t>(stream), err, g_timeout_ns, block_table, seqlens, max_pages,
                               num_pages, 1, nullptr, nullptr);
    if (rc == FA_ERR_CUDA) cuda_fail(cudaGetLastError());
    return static_cast<fa_status>(rc);
  }
  int n = num_splits;
  if (n == 0) {
    const int sms = sm_count();
    if (!sms) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
    n = fa_decode_num_splits(B, Hq, Hkv, T, max_pages * page_size, 1, sms);
  }
  if (n > 1) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID_ARG;
    if (ws_bytes < fa_decode_workspace_bytes(B, Hq, T, d, n)) return FA_ERR_INVALID_ARG;
  }
  unsigned* err = error_word();
  if (!err) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
  int rc = launch_decode(q, k_pages, v_pages, block_table, seqlens, o, lse, B, Hq, Hkv, T, 0, max_pages, num_pages, d,
                         scale, causal ? 1 : 0, n, workspace, static_cast<cudaStream_t>(stream), err, g_timeout_ns);
  if (rc == FA_ERR_CUDA) cuda_fail(cudaGetLastError());
  return static_cast<fa_status>(rc);
}

fa_status fa_get_last_device_error(void* stream, int* detail) {
  unsigned* err = error_word();
  if (!err) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return static_cast<fa_status>(cuda_fail(e));
  unsigned word = 0;
  e = cudaMemcpy(&word, err, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return static_cast<fa_status>(cuda_fail(e));
  const unsigned zero = 0;
  e = cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return static_cast<fa_status>(cuda_fail(e));
  if (detail) *detail = static_cast<int>(word);
  const unsigned code = word & 0xffu;
  if (code == 0) return FA_OK;
  return (code == FA_ERR_TIMEOUT || code == FA_ERR_BOUNDS) ? static_cast<fa_status>(code) : FA_ERR_CUDA;
}

fa_status fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream) {
  unsigned* err = error_word();
  if (!err) return static_cast<fa_status>(cuda_fail(cudaGetLastError()));
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, timeout_ns);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FA_OK : static_cast<fa_status>(cuda_fail(e));
}

}  // extern "C"
