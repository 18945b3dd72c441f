// Rotary position embedding kernels outside the attention kernels:
//   rope_rotate_kernel   y = rotate(x) for a [BH, S, D] bf16 tensor (HBM-bound), used for the
//                        operand that the attention kernel re-reads from many CTAs (K in the
//                        forward, Q in the backward), so that it is rotated once, not per load;
//   rope_convert_kernel  the backward's dQ: bf16(scale * unrotate(f32 accumulator)).
// The operand that the attention kernel loads exactly once per tile is rotated on load, in
// shared memory (Q in the forward, K in the backward), and dK is turned back in the epilogue
// of the backward's main kernel.
#include "common.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace gqa {
namespace {

// One thread per (row, group of 8 pairs).
__global__ void __launch_bounds__(256) rope_rotate_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ y,
                                                          const float* __restrict__ cs, const float* __restrict__ sn,
                                                          long long rows, int S, int D, int* status) {
  const int groups = D / 16;
  const long long n = rows * groups;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (long long)gridDim.x * blockDim.x) {
    const long long row = t / groups;
    const int gi = (int)(t - row * groups);
    const int p = (int)(row % S);
    const size_t base = (size_t)row * D + gi * 8;
    if (!dbg_range((long long)base, D / 2 + 8, rows * D, status) ||
        !dbg_range((long long)p * (D / 2) + gi * 8, 8, (long long)S * (D / 2), status))
      continue;
    uint4 lo = *reinterpret_cast<const uint4*>(x + base);
    uint4 hi = *reinterpret_cast<const uint4*>(x + base + D / 2);
    const float* c = cs + (size_t)p * (D / 2) + gi * 8;
    const float* s = sn + (size_t)p * (D / 2) + gi * 8;
    rope_rotate8_bf16(lo, hi, __ldg(reinterpret_cast<const float4*>(c)), __ldg(reinterpret_cast<const float4*>(c + 4)),
                      __ldg(reinterpret_cast<const float4*>(s)), __ldg(reinterpret_cast<const float4*>(s + 4)), 1.f);
    *reinterpret_cast<uint4*>(y + base) = lo;
    *reinterpret_cast<uint4*>(y + base + D / 2) = hi;
  }
}

// dQ = bf16(unrotate(scale * acc)), one thread per (row, group of 8 pairs).
__global__ void __launch_bounds__(256) rope_convert_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                                                           const float* __restrict__ cs, const float* __restrict__ sn,
                                                           long long rows, int S, int D, float scale,
                                                           int* status) {
  const int groups = D / 16;
  const long long n = rows * groups;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (long long)gridDim.x * blockDim.x) {
    const long long row = t / groups;
    const int gi = (int)(t - row * groups);
    const int p = (int)(row % S);
    const size_t base = (size_t)row * D + gi * 8;
    if (!dbg_range((long long)base, D / 2 + 8, rows * D, status) ||
        !dbg_range((long long)p * (D / 2) + gi * 8, 8, (long long)S * (D / 2), status))
      continue;
    const float4 a0 = *reinterpret_cast<const float4*>(acc + base);
    const float4 a1 = *reinterpret_cast<const float4*>(acc + base + 4);
    const float4 b0 = *reinterpret_cast<const float4*>(acc + base + D / 2);
    const float4 b1 = *reinterpret_cast<const float4*>(acc + base + D / 2 + 4);
    const float4 c0 = __ldg(reinterpret_cast<const float4*>(cs + (size_t)p * (D / 2) + gi * 8));
    const float4 c1 = __ldg(reinterpret_cast<const float4*>(cs + (size_t)p * (D / 2) + gi * 8 + 4));
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(sn + (size_t)p * (D / 2) + gi * 8));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(sn + (size_t)p * (D / 2) + gi * 8 + 4));
    const float x[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float y[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int i = 2 * w;
      lo[w] = pack_bf16(scale * (x[i] * c[i] + y[i] * s[i]), scale * (x[i + 1] * c[i + 1] + y[i + 1] * s[i + 1]));
      hi[w] = pack_bf16(scale * (y[i] * c[i] - x[i] * s[i]), scale * (y[i + 1] * c[i + 1] - x[i + 1] * s[i + 1]));
    }
    *reinterpret_cast<uint4*>(dq + base) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(dq + base + D / 2) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  }
}

int grid_for(long long n) {
  const int sms = device_sm_count();
  const long long want = (n + 255) / 256;
  const long long cap = (long long)sms * 8;
  return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_rope_rotate(const void* x, void* y, const float* cs, const float* sn, long long rows, int S, int D,
                               int* status, cudaStream_t stream) {
  trace_begin(kKernelRope, stream);
  rope_rotate_kernel<<<grid_for(rows * (D / 16)), 256, 0, stream>>>(static_cast<const uint16_t*>(x),
                                                                    static_cast<uint16_t*>(y), cs, sn, rows, S, D,
                                                                    status);
  cudaError_t e = cudaGetLastError();
  trace_end(kKernelRope, stream);
  return e;
}

cudaError_t launch_rope_convert(const float* acc, void* dq, const float* cs, const float* sn, long long rows, int S,
                                int D, float scale, int* status, cudaStream_t stream) {
  trace_begin(kKernelBwdConvert, stream);
  rope_convert_kernel<<<grid_for(rows * (D / 16)), 256, 0, stream>>>(acc, static_cast<uint16_t*>(dq), cs, sn, rows,
                                                                     S, D, scale, status);
  cudaError_t e = cudaGetLastError();
  trace_end(kKernelBwdConvert, stream);
  return e;
}

}  // namespace gqa
