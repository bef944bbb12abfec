// Allocation-free variant of the split-K attention operator.
//
// Some callers may not allocate device memory once they are running: a
// serving loop whose device memory budget is fixed at start-up, or a host
// thread that must not trigger the device-wide synchronisation that
// cudaMalloc / cudaFree can cause.  tqd_op_attention needs caller-provided
// scratch for its per-chunk partial results; this variant keeps that scratch
// in a fixed-size array in the library's own device image instead, so the
// caller passes only inputs and outputs and nothing is allocated per call.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "tqd.h"
#include "tqd_internal.h"

using namespace tqd;

namespace {

// Largest scratch the variant serves; every device that loads the library
// holds this array until the process exits.
constexpr size_t kScratchBytes = size_t(1) << 20;  // 1 MiB
constexpr int kMaxDevices = 64;

// Partial results (o, m, l) of every chunk, then one arrival counter per kv
// head.  Shared by all calls on a device; see the contract in tqd.h.
static __device__ __align__(256) unsigned char g_attention_scratch[kScratchBytes];

// The array's device address per device, looked up on first use; a failed
// lookup (for instance inside a stream capture) is not remembered, so the next
// call tries again.
std::mutex g_lookup_mu[kMaxDevices];
void* g_scratch_ptr[kMaxDevices];

cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_lookup_mu[dev]);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_attention_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t tqd_op_attention_noalloc_max_scratch(void) { return kScratchBytes; }

int32_t tqd_op_attention_noalloc(const float* q, const float* K, const float* V, int32_t S,
                                 int32_t n_heads, int32_t n_kv, int32_t head_dim, int32_t n_chunks,
                                 float* out, void* stream) {
  if (!q || !K || !V || !out || S <= 0 || n_heads <= 0 || n_kv <= 0 || n_heads % n_kv ||
      n_chunks < 1 || n_chunks > 1024 || !attention_supported(head_dim, n_heads / n_kv)) {
    set_last_error("tqd_op_attention_noalloc: bad argument");
    return TQD_ERR_BAD_ARG;
  }
  const size_t need = tqd_attention_scratch_bytes(n_heads, n_kv, head_dim, n_chunks);
  if (need > kScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof msg,
             "tqd_op_attention_noalloc: needs %zu bytes of scratch, the static array holds %zu",
             need, kScratchBytes);
    set_last_error(msg);
    return TQD_ERR_BAD_ARG;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    set_last_error("tqd_op_attention_noalloc: no usable current device");
    return e != cudaSuccess ? TQD_ERR_CUDA : TQD_ERR_NO_DEVICE;
  }
  // With this device current, the array's device address (its name in host
  // code is only a stand-in for the symbol), looked up once it succeeds.
  void* base = nullptr;
  e = scratch_address(dev, &base);
  if (e != cudaSuccess) {
    cudaGetLastError();  // the failed lookup leaves no error behind for later calls
    set_last_error("tqd_op_attention_noalloc: cudaGetSymbolAddress failed");
    return TQD_ERR_CUDA;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* po = static_cast<float*>(base);
  float* pml = po + static_cast<size_t>(n_heads) * n_chunks * head_dim;
  uint32_t* cnt = reinterpret_cast<uint32_t*>(pml + static_cast<size_t>(n_heads) * n_chunks * 2);
  // the arrival counters must start at zero (the partials are overwritten)
  e = cudaMemsetAsync(cnt, 0, sizeof(uint32_t) * n_kv, st);
  if (e == cudaSuccess)
    e = launch_op_attention(q, K, V, S, n_heads, n_kv, head_dim, n_chunks, out, po, pml, cnt, st);
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return TQD_ERR_CUDA;
  }
  return TQD_OK;
}

}  // extern "C"
