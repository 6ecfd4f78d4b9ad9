// decode_static.cu -- split-KV decode whose scratch lives in the library itself.
//
// fa_decode_splitkv needs a caller-provided workspace for the per-split
// partial outputs. Some callers cannot hand one over: code that runs while
// a CUDA graph is being captured (no allocation allowed), engines whose
// device memory is carved up once at start-up by someone else, plugins whose
// host owns every allocation, and latency-critical loops that must never
// risk an allocation failing or stalling. fa_decode_splitkv_static serves
// them: it runs the same decode and merge kernels, with the partials placed
// in a fixed device array that is part of the library image. It calls no
// cudaMalloc, cudaFree or other allocating routine.
//
// The array is kFaStaticScratchBytes (4 MiB). Every device that loads the
// library holds its own copy of it until the process exits. All calls on a
// device share it and it keeps whatever the previous call left there; each
// call writes every partial it later reads, so nothing has to start at zero.
// Two calls that run at the same time on the GPU (different streams, or
// different host threads) race on the array: serialise them.
#include <mutex>

#include "common.cuh"

namespace fa {

int launch_decode(const void* q, const void* k, const void* v, const int* block_table, const int* seqlens, void* o,
                  float* lse, int B, int Hq, int Hkv, int T, int S, int max_pages, int num_pages, int d, float scale,
                  int causal, int num_splits, void* workspace, cudaStream_t stream, unsigned* err,
                  unsigned long long timeout_ns);
unsigned* device_error_word();
unsigned long long wait_timeout_ns();
int device_sm_count();

constexpr size_t kFaStaticScratchBytes = 4u << 20;

// The scratch itself. In host code `g_fa_static_scratch` only names a host-side
// stand-in for the symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_fa_static_scratch[kFaStaticScratchBytes];

static std::mutex g_static_mu;

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached for the life of the
// process. Null on failure. A device reset (cudaDeviceReset) after the first
// call would leave the cached address dangling: it is not supported.
static void* static_scratch_address(cudaError_t* why) {
  static void* addr[128] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 128) {
    *why = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fa_static_scratch);
    if (e != cudaSuccess || !p) {
      *why = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}


}  // namespace fa

using namespace fa;

extern "C" {

fa_status fa_decode_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                   int Hkv, int T, int S, int d, float scale, int causal, int num_splits,
                                   void* stream) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al16(q) || !al16(k) || !al16(v) || !al16(o)) return FA_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || T < 1 || S < 1 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return FA_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > 1024) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((Hq / Hkv) * T > 16) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hkv > 65535 || static_cast<long long>(B) * Hkv * S >= (1ll << 31) ||
      static_cast<long long>(B) * Hq * T >= (1ll << 31))
    return FA_ERR_UNSUPPORTED;
  int n = num_splits;
  if (n == 0) {
    const int sms = device_sm_count();
    if (!sms) return static_cast<fa_status>(record_cuda_failure(cudaGetLastError()));
    n = fa_decode_num_splits(B, Hq, Hkv, T, S, 0, sms);
  }
  // partials that do not fit the fixed array are refused, never truncated
  if (fa_decode_workspace_bytes(B, Hq, T, d, n) > kFaStaticScratchBytes) return FA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (n > 1) {
    cudaError_t why = cudaSuccess;
    scratch = static_scratch_address(&why);
    if (!scratch) return static_cast<fa_status>(record_cuda_failure(why));
  }
  unsigned* err = device_error_word();
  if (!err) return static_cast<fa_status>(record_cuda_failure(cudaGetLastError()));
  int rc = launch_decode(q, k, v, nullptr, nullptr, o, lse, B, Hq, Hkv, T, S, 0, 0, d, scale, causal ? 1 : 0, n,
                         scratch, static_cast<cudaStream_t>(stream), err, wait_timeout_ns());
  if (rc == FA_ERR_CUDA) record_cuda_failure(cudaGetLastError());
  return static_cast<fa_status>(rc);
}

}  // extern "C"
