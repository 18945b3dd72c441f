// Rotary position embedding, rotate-half pairing: for position p and
// 0 <= i < D/2 the plane (x[i], x[i + D/2]) turns by the angle whose cosine and
// sine the caller's tables hold at [p, i] (tang page, "A transformer": RoPE
// with GQA attention, forward and backward; RustingBrain docs, "What is in the
// box": rotary positions). The backward turns gradients back by the transposed
// rotation (sine negated). Arithmetic in f32; bf16 results round to nearest even.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace gqa {

// Rotates 8 consecutive pairs held as bf16 in lo (x[i .. i+7]) and hi (x[i+D/2 ..]),
// with cos c[0..7] and sine sgn * s[0..7].
__device__ __forceinline__ void rope_rotate8_bf16(uint4& lo, uint4& hi, const float4& c0, const float4& c1,
                                                  const float4& s0, const float4& s1, float sgn) {
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float s[8] = {sgn * s0.x, sgn * s0.y, sgn * s0.z, sgn * s0.w,
                      sgn * s1.x, sgn * s1.y, sgn * s1.z, sgn * s1.w};
  uint32_t a[4] = {lo.x, lo.y, lo.z, lo.w};
  uint32_t b[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float x0 = __uint_as_float(a[w] << 16), x1 = __uint_as_float(a[w] & 0xFFFF0000u);
    const float y0 = __uint_as_float(b[w] << 16), y1 = __uint_as_float(b[w] & 0xFFFF0000u);
    const float ca = c[2 * w], cb = c[2 * w + 1], sa = s[2 * w], sb = s[2 * w + 1];
    a[w] = pack_bf16(x0 * ca - y0 * sa, x1 * cb - y1 * sb);
    b[w] = pack_bf16(y0 * ca + x0 * sa, y1 * cb + x1 * sb);
  }
  lo = make_uint4(a[0], a[1], a[2], a[3]);
  hi = make_uint4(b[0], b[1], b[2], b[3]);
}

// Rotates one row of a 128-byte-swizzled tile in shared memory in place: the row's
// 16-byte units (8 columns each) sit in boxes of 64 columns, 16 KB apart, unit u of row r
// at (u ^ (r & 7)) * 16 within the row's 128 bytes. Pairs (i, i + D/2) are unit u and
// unit u + D/16 at the same column offset. cs, sn: the row's table rows (D/2 floats).
// Only the pairs of units [u_begin, u_end) of the low half are turned.
template <int D>
__device__ __forceinline__ void rope_rotate_row_smem(uint8_t* tile, int r, const float* cs, const float* sn,
                                                     float sgn, int u_begin = 0, int u_end = D / 16) {
  constexpr int kHalfUnits = D / 16;  // 16-byte units per half row
  for (int u = u_begin; u < u_end; ++u) {
    const int uh = u + kHalfUnits;
    uint4* plo = reinterpret_cast<uint4*>(tile + (u >> 3) * 16384 + r * 128 + (((u & 7) ^ (r & 7)) << 4));
    uint4* phi = reinterpret_cast<uint4*>(tile + (uh >> 3) * 16384 + r * 128 + (((uh & 7) ^ (r & 7)) << 4));
    uint4 lo = *plo, hi = *phi;
    const float4 c0 = __ldg(reinterpret_cast<const float4*>(cs + 8 * u));
    const float4 c1 = __ldg(reinterpret_cast<const float4*>(cs + 8 * u + 4));
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(sn + 8 * u));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(sn + 8 * u + 4));
    rope_rotate8_bf16(lo, hi, c0, c1, s0, s1, sgn);
    *plo = lo;
    *phi = hi;
  }
}

}  // namespace gqa
