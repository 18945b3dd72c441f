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
//                   the CTA that finishes last among the chunks of its
//                   (batch, KV head) (an arrival ticket taken after a fence)
//                   merges all the partials in chunk order and writes O (bf16)
//                   and LSE (f32), so that no second kernel is launched.
//
// The work is bound by HBM (each cached key and value is read once). The key /
// value tiles are staged by TMA in the same 128B-swizzled 128-row boxes as the
// training kernels; the G Sq <= 16 query rows of a KV head are the M = 16 rows
// of mma.sync m16n8k16 bf16 products (S = Q K^T, O += P V) with operands read
// by ldmatrix: a 128-row tcgen05 tile would be at least 4x padding here, and
// the tensor work is a small fraction of the time the cache takes to stream.
#include <type_traits>

#include "common.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kDecWarps = 4;                        // compute warps; warp 4 is the TMA producer
constexpr int kDecWarpKeys = kDecodeKeys / kDecWarps;  // keys of a tile per compute warp (16)
constexpr int kDecThreads = 32 * (kDecWarps + 1);
constexpr int kDecBox = kDecodeKeys * 128;             // one 64-row box of 64 bf16 columns

template <int D>
struct DecCfg {
  static constexpr int kChunks = D / kChunk;
  static constexpr int kTileBytes = kDecodeKeys * D * 2;  // 64 keys
  static constexpr int kStages = (D == 64) ? 6 : 3;  // ~96 KB of K/V per CTA, two CTAs per SM
  static constexpr int kKOff = 0;
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
  int last;  // this CTA took the last ticket of its (batch, KV head): it merges the partials
};
static_assert(sizeof(DecBars<DecCfg<64>::kStages>) <= DecCfg<64>::kBarBytes, "decode barriers exceed their space");
static_assert(sizeof(DecBars<DecCfg<128>::kStages>) <= DecCfg<128>::kBarBytes, "decode barriers exceed their space");
static_assert(DecCfg<64>::kSmemBytes <= 232448 && DecCfg<128>::kSmemBytes <= 232448, "decode smem over the limit");

struct DecKParams {
  const uint16_t* q;   // [B, Hq, Sq, D]
  uint16_t* o;         // [B, Hq, Sq, D]
  float* lse;          // [B, Hq, Sq]
  float* part_acc;     // [B*Hkv, splits, R, D]
  float* part_ml;      // [B*Hkv, splits, R, 2]: (m, l), m in log2 units
  unsigned* tickets;   // [B*Hkv]: chunks of the (batch, KV head) finished so far (zeroed per call)
  int Hq, Hkv, Sq, Sk, causal, splits, chunk;
  float scale_log2;
  int* status;
};

// Four 8x8 b16 matrices from shared memory; lane l gives the row address of matrix l / 8.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// The same, each matrix transposed.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// d (m16n8, f32) += a (m16k16, bf16, row) * b (k16n8, bf16, col).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int D, int R>
__global__ void __launch_bounds__(kDecThreads, kDecodeCtasPerSm)
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
  const int n_tiles = key1 > key0 ? (key1 - key0 + kDecodeKeys - 1) / kDecodeKeys : 0;
  const WaitGuard wg{&bars->abort_flag, p.status, kWaitLimitNs};

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], kDecWarps);  // every compute warp, once done with the tile
    }
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // This warp's softmax state over its keys, in the m16n8 accumulator layout of mma.sync:
  // thread (lane) holds query rows r0 = lane / 4 and r0 + 8 (of the 16 rows, padding past R),
  // and, of every 8-column block, columns 2 (lane % 4) and 2 (lane % 4) + 1.
  constexpr int kNB = D / 8;  // 8-column blocks of O
  const int r0 = lane >> 2;
  const int cq = (lane & 3) * 2;
  float m[2] = {-INFINITY, -INFINITY};  // running max (log2 units) of rows r0, r0 + 8
  float l[2] = {0.f, 0.f};              // this thread's share of the row sums
  float acc[kNB][4];
#pragma unroll
  for (int nb = 0; nb < kNB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
  if (warp == kDecWarps) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int t = 0; t < n_tiles; ++t) {
        const int st = t % ST, use = t / ST;
        if (use > 0 && !mbar_wait(&bars->kv_empty[st], (use - 1) & 1, wg)) break;
        const int y = key0 + t * kDecodeKeys;
        mbar_arrive_expect_tx(&bars->k_full[st], C::kTileBytes);
        const bool kv_ok = dbg_tile(0, y, kvh, D, kChunk, 0, p.Sk, (int)gridDim.y, p.status);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d_chk(smem + C::kKOff + st * C::kTileBytes + c * kDecBox, &map_k, &bars->k_full[st], c * kChunk,
                          y, kvh, kv_ok, kDecBox);
        mbar_arrive_expect_tx(&bars->v_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d_chk(smem + C::kVOff + st * C::kTileBytes + c * kDecBox, &map_v, &bars->v_full[st], c * kChunk,
                          y, kvh, kv_ok, kDecBox);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    // Warp w takes keys [16 w, 16 w + 16) of every 64-key tile (two CTAs per SM keep the
    // cache streaming while either starts or ends). S = Q K^T and O += P V run as m16n8k16 bf16
    // MMAs (the G Sq <= 16 query rows of the KV head are the M = 16 rows), operands read from
    // the 128B-swizzled tiles with ldmatrix.
    constexpr int kWNB = kDecWarpKeys / 8;   // 8-key blocks of S per warp
    constexpr int kWKS = kDecWarpKeys / 16;  // 16-key steps of P V per warp
    const int wq = warp;
    // Q as A fragments, one per 16 columns of D (unscaled bf16; the scores are scaled in f32).
    uint32_t qa[D / 16][4];
    {
      auto qword = [&](int r, int col) -> uint32_t {  // bf16 pair (col, col + 1) of query row r
        const int hl = r / p.Sq, i = r - hl * p.Sq;
        if (r >= R || hl >= G) return 0u;  // padding rows: zero queries, partials never read
        const size_t at = (((size_t)b * p.Hq + g * G + hl) * p.Sq + i) * D + col;
        if (!dbg_range((long long)at, 2, (long long)gridDim.y / p.Hkv * p.Hq * p.Sq * D, p.status)) return 0u;
        return *reinterpret_cast<const uint32_t*>(p.q + at);
      };
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qa[ks][0] = qword(r0, 16 * ks + cq);
        qa[ks][1] = qword(r0 + 8, 16 * ks + cq);
        qa[ks][2] = qword(r0, 16 * ks + 8 + cq);
        qa[ks][3] = qword(r0 + 8, 16 * ks + 8 + cq);
      }
    }
    const float c = p.scale_log2;
    const int causal_base = p.Sk - p.Sq;  // row r sees keys <= causal_base + r % Sq
    const int vis0 = causal_base + (r0 % p.Sq), vis1 = causal_base + ((r0 + 8) % p.Sq);
    for (int t = 0; t < n_tiles; ++t) {
      const int st = t % ST;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->k_full[st], (t / ST) & 1, wg))) break;
      const uint32_t sK = smem_addr(smem + C::kKOff + st * C::kTileBytes);
      const int kb = wq * kDecWarpKeys;  // this warp's first key in the tile
      // ---- S (16 rows x 16 keys), blocks of 8 keys
      float sc[kWNB][4];
#pragma unroll
      for (int nb = 0; nb < kWNB; ++nb) {
        sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
        const int key = kb + 8 * nb + (lane & 7);  // this lane's row address for ldmatrix
#pragma unroll
        for (int ks = 0; ks < D / 16; ks += 2) {
          // four 8x8 matrices: d [16ks, +8), [16ks+8, +8), [16ks+16, +8), [16ks+24, +8) of 8 keys
          const int d0 = 16 * ks + 8 * (lane >> 3);
          const uint32_t addr = sK + (d0 >> 6) * kDecBox + key * 128 + ((((d0 & 63) >> 3) ^ (key & 7)) << 4);
          uint32_t kf[4];
          ldmatrix_x4(addr, kf);
          mma_bf16_16816(sc[nb], qa[ks], kf[0], kf[1]);
          mma_bf16_16816(sc[nb], qa[ks + 1], kf[2], kf[3]);
        }
      }
      // ---- mask (keys past the chunk / the cache; causal per row) and online softmax
      const int tkey = key0 + t * kDecodeKeys + kb;
      float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nb = 0; nb < kWNB; ++nb) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = tkey + 8 * nb + cq + (e & 1);
          const bool vis = key < key1 && (!p.causal || key <= ((e & 2) ? vis1 : vis0));
          sc[nb][e] = vis ? sc[nb][e] * c : -INFINITY;
          mt[e >> 1] = fmaxf(mt[e >> 1], sc[nb][e]);
        }
      }
      float alpha[2], ref[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 1));
        mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 2));
        const float mn = fmaxf(m[h], mt[h]);
        ref[h] = (mn == -INFINITY) ? 0.f : mn;  // no visible key yet: keep the state empty
        alpha[h] = ex2_approx(m[h] - ref[h]);   // 0 when m was -inf
        m[h] = mn;
        l[h] *= alpha[h];
      }
#pragma unroll
      for (int nb = 0; nb < kNB; ++nb) {
        acc[nb][0] *= alpha[0];
        acc[nb][1] *= alpha[0];
        acc[nb][2] *= alpha[1];
        acc[nb][3] *= alpha[1];
      }
      // P (bf16) as the A fragments of the 16-key steps
      uint32_t pa[kWKS][4];
#pragma unroll
      for (int nb = 0; nb < kWNB; ++nb) {
        const float p0 = ex2_approx(sc[nb][0] - ref[0]), p1 = ex2_approx(sc[nb][1] - ref[0]);
        const float p2 = ex2_approx(sc[nb][2] - ref[1]), p3 = ex2_approx(sc[nb][3] - ref[1]);
        l[0] += p0 + p1;
        l[1] += p2 + p3;
        pa[nb >> 1][(nb & 1) * 2] = pack_bf16(p0, p1);
        pa[nb >> 1][(nb & 1) * 2 + 1] = pack_bf16(p2, p3);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[st], (t / ST) & 1, wg))) break;
      const uint32_t sV = smem_addr(smem + C::kVOff + st * C::kTileBytes);
      // ---- O += P V: per 16 keys and pair of 8-column blocks, four transposed 8x8 matrices
#pragma unroll
      for (int kp = 0; kp < kWKS; ++kp) {
        const int key = kb + 16 * kp + 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
        for (int nb = 0; nb < kNB; nb += 2) {
          const int d0 = 8 * (nb + (lane >> 4));
          const uint32_t addr = sV + (d0 >> 6) * kDecBox + key * 128 + ((((d0 & 63) >> 3) ^ (key & 7)) << 4);
          uint32_t vf[4];
          ldmatrix_x4_trans(addr, vf);
          mma_bf16_16816(acc[nb], pa[kp], vf[0], vf[1]);
          mma_bf16_16816(acc[nb + 1], pa[kp], vf[2], vf[3]);
        }
      }
      mbar_arrive_warp(&bars->kv_empty[st]);
    }
    // row sums: this thread's share over its columns, then over the 4 threads of the row
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
    }
  }
  // The combine buffer overlays the K/V ring: every warp must be done with its tiles first.
  __syncthreads();
  if (warp < kDecWarps) {
    // ---- this warp's state of each real row (r < R) into the combine buffer
    float* red = reinterpret_cast<float*>(smem + C::kRedOff);  // [warp][R][D + 2]
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = r0 + 8 * h;
      if (r < R) {
        float* dst = red + (warp * R + r) * (D + 2);
#pragma unroll
        for (int nb = 0; nb < kNB; ++nb) {
          dst[8 * nb + cq] = acc[nb][2 * h];
          dst[8 * nb + cq + 1] = acc[nb][2 * h + 1];
        }
        if ((lane & 3) == 0) {
          dst[D] = m[h];
          dst[D + 1] = l[h];
        }
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
    if (!dbg_range((long long)pr_row, 1, (long long)gridDim.y * p.splits * R, p.status)) continue;
    p.part_acc[pr_row * D + d] = a;
    if (d == 0) {
      p.part_ml[pr_row * 2] = M;
      p.part_ml[pr_row * 2 + 1] = L;
    }
  }

  // ---- arrival ticket: the last chunk of this (batch, KV head) to finish merges all partials.
  // The barrier orders every thread's partial stores before thread 0's fence, which (being
  // cumulative) makes them visible device-wide before its ticket; the last CTA's thread 0
  // fences after reading the ticket and the barrier hands that on to the CTA's other threads.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    bars->last = dbg_ok(kvh < (int)gridDim.y && (int)gridDim.x == p.splits, p.status) &&
                         atomicAdd(p.tickets + kvh, 1u) == (unsigned)p.splits - 1u
                     ? 1
                     : 0;
    __threadfence();
  }
  __syncthreads();
  if (!bars->last) return;
  // One warp per real query row r = (h % G) Sq + i of the group: lane s holds chunk s's (m, l)
  // (chunks past 32 in further rounds), the lanes hold the accumulator's columns; the first
  // kPre chunks' accumulators are loaded in the same round trip as the (m, l) pairs. The max
  // and the sum of l use a fixed shuffle order and the accumulator takes the chunks in order,
  // so the result does not depend on which CTA arrived last. Partials are read from L2.
  constexpr int kDC = D / 32;
  constexpr int kPre = 8;
  using Vec = typename std::conditional<kDC == 4, float4, float2>::type;
  for (int r = warp; r < G * p.Sq; r += kDecThreads / 32) {
    const size_t row0 = (size_t)kvh * p.splits * R + r;  // partial row of chunk s: row0 + s R
    Vec pre[kPre];
#pragma unroll
    for (int s = 0; s < kPre; ++s)
      if (s < p.splits) pre[s] = __ldcg(reinterpret_cast<const Vec*>(p.part_acc + (row0 + (size_t)s * R) * D) + lane);
    float2 mine = make_float2(-INFINITY, 0.f);  // (m, l) of chunk `lane` (splits <= 32)
    if (lane < p.splits) mine = __ldcg(reinterpret_cast<const float2*>(p.part_ml + (row0 + (size_t)lane * R) * 2));
    float M = mine.x;
    for (int s = lane + 32; s < p.splits; s += 32) M = fmaxf(M, __ldcg(p.part_ml + (row0 + (size_t)s * R) * 2));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float ref = (M == -INFINITY) ? 0.f : M;
    const float f_mine = ex2_approx(mine.x - ref);  // 0 for lanes past the chunks
    float L = mine.y * f_mine;
    for (int s = lane + 32; s < p.splits; s += 32) {
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + (row0 + (size_t)s * R) * 2));
      L = fmaf(ml.y, ex2_approx(ml.x - ref), L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float acc_o[kDC];
#pragma unroll
    for (int c = 0; c < kDC; ++c) acc_o[c] = 0.f;
    auto add = [&](const Vec& v, float f) {
      if constexpr (kDC == 4) {
        acc_o[0] = fmaf(v.x, f, acc_o[0]);
        acc_o[1] = fmaf(v.y, f, acc_o[1]);
        acc_o[2] = fmaf(v.z, f, acc_o[2]);
        acc_o[3] = fmaf(v.w, f, acc_o[3]);
      } else {
        acc_o[0] = fmaf(v.x, f, acc_o[0]);
        acc_o[1] = fmaf(v.y, f, acc_o[1]);
      }
    };
#pragma unroll
    for (int s = 0; s < kPre; ++s)
      if (s < p.splits) add(pre[s], __shfl_sync(0xffffffffu, f_mine, s));
#pragma unroll 4
    for (int s = kPre; s < p.splits; ++s) {
      const size_t pr = row0 + (size_t)s * R;
      const float f = s < 32 ? __shfl_sync(0xffffffffu, f_mine, s & 31) : ex2_approx(__ldcg(p.part_ml + pr * 2) - ref);
      add(__ldcg(reinterpret_cast<const Vec*>(p.part_acc + pr * D) + lane), f);
    }
    const float inv = 1.f / L;
    const int h = g * G + r / p.Sq;
    const int i = r - (r / p.Sq) * p.Sq;
    const size_t orow = ((size_t)b * p.Hq + h) * p.Sq + i;
    if (!dbg_range((long long)orow, 1, (long long)gridDim.y / p.Hkv * p.Hq * p.Sq, p.status)) continue;
    uint16_t* op = p.o + orow * D + lane * kDC;
    if constexpr (kDC == 4) {
      *reinterpret_cast<uint2*>(op) =
          make_uint2(pack_bf16(acc_o[0] * inv, acc_o[1] * inv), pack_bf16(acc_o[2] * inv, acc_o[3] * inv));
    } else {
      *reinterpret_cast<uint32_t*>(op) = pack_bf16(acc_o[0] * inv, acc_o[1] * inv);
    }
    if (lane == 0) p.lse[orow] = (M + __log2f(L)) * 0.69314718055994530942f;
  }
}

template <int D, int R>
cudaError_t launch_split(const DecodeArgs& a, const DecKParams& p, cudaStream_t stream) {
  using C = DecCfg<D>;
  cudaError_t e = kernel_setup(reinterpret_cast<const void*>(decode_split_kernel<D, R>), C::kSmemBytes,
                               kDecThreads, 0);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.splits, (unsigned)(a.B * a.Hkv));
  decode_split_kernel<D, R><<<grid, kDecThreads, C::kSmemBytes, stream>>>(*a.map_k, *a.map_v, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs& a, cudaStream_t stream) {
  DecKParams p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.o = static_cast<uint16_t*>(a.o);
  p.lse = a.lse;
  p.part_acc = a.part_acc;
  p.part_ml = a.part_ml;
  p.tickets = a.tickets;
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
  // The tickets start from zero on every call (the caller's workspace holds them).
  cudaError_t e = cudaMemsetAsync(a.tickets, 0, sizeof(unsigned) * (size_t)a.B * a.Hkv, stream);
  if (e != cudaSuccess) return e;
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
  return e;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.D == 64) return launch_decode_d<64>(a, stream);
  return launch_decode_d<128>(a, stream);
}

}  // namespace gqa
