// Attention of a few new queries against a key/value cache (decode), split over
// key chunks and recombined with the online-softmax monoid.
//
// The pages' KV-cached decoding (RustingBrain docs, "Training infrastructure";
// tang page, "An LLM": decode at 4k context) attends Sq new query rows to Sk
// cached keys; new query i sits at absolute position Sk - Sq + i and, causal,
// sees keys j <= Sk - Sq + i. Because the softmax state (m, l, acc) combines
// associatively (tang page, "How tang works", section 3, last paragraph), the
// keys are split into chunks processed by different CTAs, and the chunk states
// are merged afterwards:
//
//   decode_split    one CTA per (batch, KV head, key chunk): the state of
//                   every query row of the KV head's group (G heads x Sq rows,
//                   R <= 16 rows) over the chunk's keys, written as a partial;
//   decode_combine  one warp per query row: merges the partials of all chunks,
//                   writes O (bf16) and LSE (f32).
//
// The work is bound by HBM (each cached key and value is read once), so the
// arithmetic runs on the CUDA cores; the key/value tiles are staged by TMA in
// the same 128B-swizzled 128-row boxes as the training kernels.
#include "common.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kDecWarps = 8;              // compute warps (two groups of 4); warp 8 is the TMA producer
constexpr int kDecGroupWarps = 4;         // warps of a group: one 128-key tile, one key per lane
constexpr int kDecThreads = 32 * (kDecWarps + 1);

template <int D>
struct DecCfg {
  static constexpr int kChunks = D / kChunk;
  static constexpr int kTileBytes = kTile * D * 2;   // 128 keys
  static constexpr int kStages = (D == 64) ? 6 : 3;  // ~192 KB of K/V in flight per CTA
  static constexpr int kDC = D / 32;                 // head-dim columns per lane in P.V
  static constexpr int kQOff = 0;                    // f32 [kMaxRows][D], pre-scaled by scale*log2(e)
  static constexpr int kKOff = kMaxDecodeRows * D * 4;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  // warp states for the final combine, over the K/V ring (every tile has been consumed by then)
  static constexpr int kRedOff = kKOff;
  static constexpr int kRedBytes = kDecWarps * kMaxDecodeRows * (D + 2) * 4;
  static_assert(kRedBytes <= 2 * kStages * kTileBytes, "combine buffer must fit in the K/V ring");
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kBarBytes = 256;  // DecBars<kStages>, checked below
  static constexpr int kSmemBytes = kBarOff + kBarBytes;
};

template <int ST>
struct DecBars {
  uint64_t k_full[ST], v_full[ST], kv_empty[ST];
  int abort_flag;
};
static_assert(sizeof(DecBars<DecCfg<64>::kStages>) <= DecCfg<64>::kBarBytes, "decode barriers exceed their space");
static_assert(sizeof(DecBars<DecCfg<128>::kStages>) <= DecCfg<128>::kBarBytes, "decode barriers exceed their space");
static_assert(DecCfg<64>::kSmemBytes <= 232448 && DecCfg<128>::kSmemBytes <= 232448, "decode smem over the limit");

struct DecKParams {
  const uint16_t* q;   // [B, Hq, Sq, D]
  float* part_acc;     // [B*Hkv, splits, R, D]
  float* part_ml;      // [B*Hkv, splits, R, 2]: (m, l), m in log2 units
  int Hq, Hkv, Sq, Sk, causal, splits, chunk;
  float scale_log2;
  int* status;
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int D, int R>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                        const DecKParams p) {
  using C = DecCfg<D>;
  constexpr int ST = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  auto* bars = reinterpret_cast<DecBars<ST>*>(smem + C::kBarOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_addr(smem) & 1023u) != 0) {
    if (tid == 0) atomicOr(p.status, STATUS_MISALIGNED_SMEM);
    return;
  }
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;  // b * Hkv + g
  const int G = p.Hq / p.Hkv;
  const int b = kvh / p.Hkv;
  const int g = kvh - b * p.Hkv;
  const int key0 = split * p.chunk;
  const int key1 = min(p.Sk, key0 + p.chunk);
  const int n_tiles = key1 > key0 ? (key1 - key0 + kTile - 1) / kTile : 0;
  const WaitGuard wg{&bars->abort_flag, p.status, kWaitLimitNs};

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], kDecGroupWarps);  // the group that consumed the tile
    }
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  // Query rows r = hl * Sq + i (hl: head within the group) as f32, pre-scaled by scale*log2(e).
  float* sq = reinterpret_cast<float*>(smem + C::kQOff);
  for (int e = tid; e < R * D; e += kDecThreads) {
    const int r = e / D, d = e - r * D;
    const int hl = r / p.Sq, i = r - hl * p.Sq;
    float x = 0.f;  // rows padded past G * Sq stay zero (their partials are never read)
    if (hl < G) x = __uint_as_float((uint32_t)p.q[(((size_t)b * p.Hq + g * G + hl) * p.Sq + i) * D + d] << 16);
    sq[e] = x * p.scale_log2;
  }
  __syncthreads();

  // this warp's softmax state over its keys (compute warps only)
  float m[R], l[R], acc[R][C::kDC];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < C::kDC; ++c) acc[r][c] = 0.f;
  }
  if (warp == kDecWarps) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int t = 0; t < n_tiles; ++t) {
        const int st = t % ST, use = t / ST;
        if (use > 0 && !mbar_wait(&bars->kv_empty[st], (use - 1) & 1, wg)) break;
        const int y = key0 + t * kTile;
        mbar_arrive_expect_tx(&bars->k_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem + C::kKOff + st * C::kTileBytes + c * kBoxBytes, &map_k, &bars->k_full[st], c * kChunk,
                      y, kvh);
        mbar_arrive_expect_tx(&bars->v_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem + C::kVOff + st * C::kTileBytes + c * kBoxBytes, &map_v, &bars->v_full[st], c * kChunk,
                      y, kvh);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    // Two groups of 4 warps take alternate tiles (two tiles in flight); each warp keeps its own
    // state, and all are merged below.
    const int grp = warp / kDecGroupWarps;
    const int wq = warp - grp * kDecGroupWarps;
    const int kk = wq * 32 + lane;  // this lane's key within a 128-key tile (scores)
    for (int t = grp; t < n_tiles; t += kDecWarps / kDecGroupWarps) {
      const int st = t % ST;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->k_full[st], (t / ST) & 1, wg))) break;
      const uint8_t* sK = smem + C::kKOff + st * C::kTileBytes;
      // ---- scores of key kk against every row
      float s[R];
#pragma unroll
      for (int r = 0; r < R; ++r) s[r] = 0.f;
#pragma unroll 4
      for (int c = 0; c < D / 8; ++c) {  // 16-byte units of the key row (8 bf16)
        const uint4 w = *reinterpret_cast<const uint4*>(sK + (c >> 3) * kBoxBytes + kk * 128 +
                                                         (((c & 7) ^ (kk & 7)) << 4));
        const float kv8[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                              bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4 qa = *reinterpret_cast<const float4*>(sq + r * D + c * 8);
          const float4 qb = *reinterpret_cast<const float4*>(sq + r * D + c * 8 + 4);
          s[r] = fmaf(qa.x, kv8[0], s[r]);
          s[r] = fmaf(qa.y, kv8[1], s[r]);
          s[r] = fmaf(qa.z, kv8[2], s[r]);
          s[r] = fmaf(qa.w, kv8[3], s[r]);
          s[r] = fmaf(qb.x, kv8[4], s[r]);
          s[r] = fmaf(qb.y, kv8[5], s[r]);
          s[r] = fmaf(qb.z, kv8[6], s[r]);
          s[r] = fmaf(qb.w, kv8[7], s[r]);
        }
      }
      // ---- mask: keys past the chunk / the cache, and (causal) past each row's position
      const int key = key0 + t * kTile + kk;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int i = r % p.Sq;
        const bool vis = key < key1 && (!p.causal || key <= p.Sk - p.Sq + i);
        if (!vis) s[r] = -INFINITY;
      }
      // ---- online-softmax update of this warp's state (log2 units)
      float pr[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float mt = warp_max(s[r]);
        const float mn = fmaxf(m[r], mt);
        const float ref = (mn == -INFINITY) ? 0.f : mn;  // no visible key yet: keep the state empty
        const float alpha = ex2_approx(m[r] - ref);       // 0 when m was -inf
        pr[r] = ex2_approx(s[r] - ref);
        l[r] = l[r] * alpha + warp_sum(pr[r]);
        m[r] = mn;
#pragma unroll
        for (int c = 0; c < C::kDC; ++c) acc[r][c] *= alpha;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[st], (t / ST) & 1, wg))) break;
      const uint8_t* sV = smem + C::kVOff + st * C::kTileBytes;
      // ---- acc += P V over this warp's 32 keys; lane owns columns [lane*kDC, lane*kDC + kDC)
      const int col0 = lane * C::kDC;
#pragma unroll 4
      for (int j = 0; j < 32; ++j) {
        const int vk = wq * 32 + j;
        const uint8_t* vrow = sV + (col0 >> 6) * kBoxBytes + vk * 128;
        const int unit = (col0 & 63) >> 3;
        const uint8_t* vp = vrow + ((unit ^ (vk & 7)) << 4) + (col0 & 7) * 2;
        float vv[C::kDC];
        if constexpr (C::kDC == 4) {
          const uint2 w = *reinterpret_cast<const uint2*>(vp);
          vv[0] = bf16_lo(w.x);
          vv[1] = bf16_hi(w.x);
          vv[2] = bf16_lo(w.y);
          vv[3] = bf16_hi(w.y);
        } else {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(vp);
          vv[0] = bf16_lo(w);
          vv[1] = bf16_hi(w);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float pj = __shfl_sync(0xffffffffu, pr[r], j);
#pragma unroll
          for (int c = 0; c < C::kDC; ++c) acc[r][c] = fmaf(pj, vv[c], acc[r][c]);
        }
      }
      mbar_arrive_warp(&bars->kv_empty[st]);
    }
  }
  // The combine buffer overlays the K/V ring: every warp must be done with its tiles first.
  __syncthreads();
  if (warp < kDecWarps) {
    // ---- combine the warps' states (same monoid) and write this chunk's partial
    float* red = reinterpret_cast<float*>(smem + C::kRedOff);  // [warp][R][D + 2]
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float* dst = red + (warp * R + r) * (D + 2);
#pragma unroll
      for (int c = 0; c < C::kDC; ++c) dst[lane * C::kDC + c] = acc[r][c];
      if (lane == 0) {
        dst[D] = m[r];
        dst[D + 1] = l[r];
      }
    }
  }
  __syncthreads();
  // threads of the CTA: one (row, column) pair per step
  for (int e = tid; e < R * D; e += kDecThreads) {
    const int r = e / D, d = e - r * D;
    const float* red = reinterpret_cast<const float*>(smem + C::kRedOff);
    float M = -INFINITY;
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, red[(w * R + r) * (D + 2) + D]);
    const float ref = (M == -INFINITY) ? 0.f : M;
    float a = 0.f, L = 0.f;
    for (int w = 0; w < kDecWarps; ++w) {
      const float* st = red + (w * R + r) * (D + 2);
      const float f = ex2_approx(st[D] - ref);
      a = fmaf(st[d], f, a);
      L = fmaf(st[D + 1], f, L);
    }
    const size_t pr_row = ((size_t)kvh * p.splits + split) * R + r;
    p.part_acc[pr_row * D + d] = a;
    if (d == 0) {
      p.part_ml[pr_row * 2] = M;
      p.part_ml[pr_row * 2 + 1] = L;
    }
  }
}

// One warp per query row (b, h, i): merge the chunk partials of its KV head group.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const float* __restrict__ part_acc,
                                                             const float* __restrict__ part_ml, uint16_t* __restrict__ o,
                                                             float* __restrict__ lse, int B, int Hq, int Hkv, int Sq,
                                                             int splits, int R) {
  constexpr int kDC = D / 32;
  const int lane = threadIdx.x & 31;
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // (b * Hq + h) * Sq + i
  if (row >= B * Hq * Sq) return;
  const int i = row % Sq;
  const int bh = row / Sq;
  const int b = bh / Hq, h = bh - b * Hq;
  const int G = Hq / Hkv;
  const int kvh = b * Hkv + h / G;
  const int r = (h % G) * Sq + i;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part_ml[(((size_t)kvh * splits + s) * R + r) * 2]);
  const float ref = (M == -INFINITY) ? 0.f : M;
  float a[kDC] = {};
  float L = 0.f;
  for (int s = 0; s < splits; ++s) {
    const size_t pr_row = ((size_t)kvh * splits + s) * R + r;
    const float f = ex2_approx(part_ml[pr_row * 2] - ref);
    L = fmaf(part_ml[pr_row * 2 + 1], f, L);
#pragma unroll
    for (int c = 0; c < kDC; ++c) a[c] = fmaf(part_acc[pr_row * D + lane * kDC + c], f, a[c]);
  }
  const float inv = 1.f / L;
  uint16_t* orow = o + (size_t)row * D + lane * kDC;
  if constexpr (kDC == 4) {
    *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16(a[0] * inv, a[1] * inv), pack_bf16(a[2] * inv, a[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(orow) = pack_bf16(a[0] * inv, a[1] * inv);
  }
  if (lane == 0) lse[row] = (M + __log2f(L)) * 0.69314718055994530942f;
}

template <int D, int R>
cudaError_t launch_split(const DecodeArgs& a, const DecKParams& p, cudaStream_t stream) {
  using C = DecCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.splits, (unsigned)(a.B * a.Hkv));
  decode_split_kernel<D, R><<<grid, kDecThreads, C::kSmemBytes, stream>>>(*a.map_k, *a.map_v, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs& a, cudaStream_t stream) {
  DecKParams p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.part_acc = a.part_acc;
  p.part_ml = a.part_ml;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.causal = a.causal;
  p.splits = a.splits;
  p.chunk = a.chunk;
  p.scale_log2 = a.scale_log2;
  p.status = a.status;
  const int R = a.Sq * (a.Hq / a.Hkv);
  cudaError_t e;
  trace_begin(kKernelDecodeSplit, stream);
  if (R <= 1)
    e = launch_split<D, 1>(a, p, stream);
  else if (R <= 2)
    e = launch_split<D, 2>(a, p, stream);
  else if (R <= 4)
    e = launch_split<D, 4>(a, p, stream);
  else if (R <= 8)
    e = launch_split<D, 8>(a, p, stream);
  else
    e = launch_split<D, 16>(a, p, stream);
  trace_end(kKernelDecodeSplit, stream);
  if (e != cudaSuccess) return e;
  const int Rpad = R <= 1 ? 1 : R <= 2 ? 2 : R <= 4 ? 4 : R <= 8 ? 8 : 16;
  const int rows = a.B * a.Hq * a.Sq;
  trace_begin(kKernelDecodeCombine, stream);
  decode_combine_kernel<D><<<(rows * 32 + 255) / 256, 256, 0, stream>>>(a.part_acc, a.part_ml,
                                                                         static_cast<uint16_t*>(a.o), a.lse, a.B,
                                                                         a.Hq, a.Hkv, a.Sq, a.splits, Rpad);
  e = cudaGetLastError();
  trace_end(kKernelDecodeCombine, stream);
  return e;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.D == 64) return launch_decode_d<64>(a, stream);
  return launch_decode_d<128>(a, stream);
}

}  // namespace gqa
