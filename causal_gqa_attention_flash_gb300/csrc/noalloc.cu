// Backward entry point that allocates nothing and takes no workspace.
//
// Some callers cannot call cudaMalloc: code that runs inside a region where
// allocation is forbidden or unsafe (a custom allocator's own callbacks, a
// framework that owns all device memory and hands out only tensors, embedded
// or real-time hosts that must not allocate after start-up). For them this
// file keeps the backward's scratch memory -- the per-row D and scaled-LSE
// arrays and the f32 dQ accumulator -- in one file-scope device array, so the
// caller passes only inputs and outputs.
//
// The array is GQA_NOALLOC_SCRATCH_BYTES (64 MiB) on every device that loads
// the library, held until the process exits. Every call on a device shares it
// and it keeps the last call's contents; the backward's prep kernel writes
// every part that must start at zero or be rewritten before it is read, so a
// call never sees the previous call's values. Calls that overlap on the GPU
// (two streams, or two host threads, at once) race on the array.
#include <mutex>

#include "../../include/gqa_attn.h"
#include "common.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GQA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and passed to the kernels.
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int gqa_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S,
                                    int D, int causal, float scale, void* stream) {
  // The codes gqa_attn_bwd itself returns for null pointers and rejected sizes or scales.
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return GQA_ERR_INVALID_ARG;
  const int rc = gqa::check_common(B, Hq, Hkv, S, D, scale);
  if (rc != GQA_OK) return rc;
  const size_t need = gqa_attn_bwd_workspace_size(B, Hq, Hkv, S, D);
  if (need > (size_t)GQA_NOALLOC_SCRATCH_BYTES) return GQA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const cudaError_t e = noalloc_scratch(&scratch);
  if (e != cudaSuccess) return gqa::record_cuda_error(e);
  return gqa_attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, scratch, (size_t)GQA_NOALLOC_SCRATCH_BYTES, B, Hq, Hkv, S, D,
                      causal, scale, stream);
}
