// Query-major dQ of fused causal grouped-query attention on sm_103a: the
// deterministic alternative to the KV-major kernel's f32 reduce-add of dQ
// partials. The backward is itself a comprehension with no S x S intermediate
// (aiinsiders.net, "A compiler that derives GPU kernels matches hand-tuned
// code"); here it is evaluated per query tile:
//
//   for every key tile j the query tile can see, in order:
//     S   = Q K_j^T,   P = exp2(S c - LSE2)      (P recomputed from the LSE)
//     dP  = dO V_j^T,  dS = P (dP - D)
//     dQ += dS K_j                               (f32, in TMEM)
//   dQ = scale * dQ -> bf16
//
// Every dQ row is summed by one CTA in a fixed order, so dQ is bitwise
// reproducible. It costs two contractions per (query, key) pair more than the
// KV-major kernel's dQ (S and dP are recomputed here; that kernel then skips
// its dQ), 14 D flops per pair for the whole backward instead of 10 D.
//
// One CTA = one (batch, query head, 128-row query tile). Keys stream in 64-row
// units u (keys 64u .. 64u+63), which alternate between two element-wise
// warpgroups: while warpgroup u % 2 works on unit u, the tensor core runs
// dQ(u-1) and S, dP of unit u+1. The K/V ring holds units, so a unit's copy is
// issued two units before its first MMA.
// Warp roles (320 threads):
//   warps 0..3  element-wise, even units: thread r owns query row r (TMEM lane r);
//   warps 4..7  element-wise, odd units;
//   warp 8      TMA producer: Q and dO once, then K and V units into a ring of stages;
//   warp 9      MMA issuer (one thread) and TMEM owner.
// TMEM columns: warpgroup h: S [128h, 128h+64) (then dS, packed bf16, in its
// first 32 columns), dP [128h+64, 128h+128); dQ [256, 256+D).
// Epilogue: dQ * scale in bf16 into the (no longer read) Q buffer in the TMA box
// layout, stored by TMA; rows past S are clipped.
#include "common.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kUnit = 64;                       // keys per unit
constexpr int kUnitBox = kUnit * 128;           // one 64-row box of 64 bf16 columns (8 KB)

template <int D>
struct DqCfg {
  static constexpr int kChunks = D / kChunk;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kUnitBytes = kUnit * D * 2;  // one unit of K (or V)
  static constexpr int kStages = (D == 64) ? 6 : 4;
  static constexpr int kQOff = 0;  // Q, then the dQ staging
  static constexpr int kDOOff = kQOff + kTileBytes;
  static constexpr int kKOff = kDOOff + kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kUnitBytes;
  static constexpr int kBarOff = kVOff + kStages * kUnitBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers + alignment slack
  static constexpr int kThreads = 320;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kDQCol = 256;
};

template <int ST>
struct DqBars {
  uint64_t qdo_full;
  uint64_t k_full[ST];
  uint64_t v_full[ST];
  uint64_t kv_empty[ST];
  uint64_t s_full[2];
  uint64_t dp_full[2];
  uint64_t ds_full[2];
  uint64_t dq_done;
  uint64_t drain;
  uint64_t epi_bar;
  uint32_t tmem_base;
  int abort_flag;
};

static_assert(sizeof(DqBars<DqCfg<64>::kStages>) <= 256 && sizeof(DqBars<DqCfg<128>::kStages>) <= 256,
              "dQ kernel barriers exceed the 256 bytes reserved for them");
static_assert(DqCfg<64>::kSmemBytes <= 232448 && DqCfg<128>::kSmemBytes <= 232448, "dQ kernel smem over the limit");

struct DqKParams {
  const float* lse2;  // f32 [B*Hq, S_pad]: LSE * log2(e), +inf past S
  const float* dvec;  // f32 [B*Hq, S_pad]: D_i = rowsum(dO * O)
  int Hq, Hkv, S, S_pad, causal;
  float scale, scale_log2;
  int* status;
};

__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

template <int D>
__global__ void __launch_bounds__(320, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                  const __grid_constant__ CUtensorMap map_dq, const DqKParams p) {
  using C = DqCfg<D>;
  constexpr int ST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  auto* bars = reinterpret_cast<DqBars<ST>*>(smem + C::kBarOff);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int bh = blockIdx.x;                            // b * Hq + h
  const int qt = (int)gridDim.y - 1 - (int)blockIdx.y;  // longest query tiles first
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int kvh = b * p.Hkv + h / (p.Hq / p.Hkv);
  // key units this query tile visits: causal, keys up to the tile's last row; else all S keys
  const int n_units = p.causal ? 2 * (qt + 1) : (p.S + kUnit - 1) / kUnit;
  const WaitGuard wg{&bars->abort_flag, p.status, kWaitLimitNs};

  if (tid == 0) {
    mbar_init(&bars->qdo_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->dp_full[i], 1);
      mbar_init(&bars->ds_full[i], 4);  // one arrival per warp of the half's warpgroup
    }
    mbar_init(&bars->dq_done, 1);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->epi_bar, 8);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_do);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      mbar_arrive_expect_tx(&bars->qdo_full, 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(smem + C::kQOff + c * kBoxBytes, &map_q, &bars->qdo_full, c * kChunk, qt * kTile, bh);
        tma_load_3d(smem + C::kDOOff + c * kBoxBytes, &map_do, &bars->qdo_full, c * kChunk, qt * kTile, bh);
      }
      int issued = 0;
      for (int u = 0; u < n_units; ++u) {
        const int st = u % ST;
        const int use = u / ST;
        if (use > 0 && !mbar_wait(&bars->kv_empty[st], (use - 1) & 1, wg)) break;
        mbar_arrive_expect_tx(&bars->k_full[st], C::kUnitBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem + C::kKOff + st * C::kUnitBytes + c * kUnitBox, &map_k, &bars->k_full[st], c * kChunk,
                      u * kUnit, kvh);
        mbar_arrive_expect_tx(&bars->v_full[st], C::kUnitBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem + C::kVOff + st * C::kUnitBytes + c * kUnitBox, &map_v, &bars->v_full[st], c * kChunk,
                      u * kUnit, kvh);
        issued = u + 1;
      }
      if (bars->abort_flag) {
        // Let every copy already issued land before the CTA's shared memory goes away.
        mbar_wait_drain(&bars->qdo_full, 0, kWaitLimitNs);
        for (int u = (issued > ST ? issued - ST : 0); u < issued; ++u) {
          mbar_wait_drain(&bars->k_full[u % ST], (u / ST) & 1, kWaitLimitNs);
          mbar_wait_drain(&bars->v_full[u % ST], (u / ST) & 1, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, kUnit, false, false);  // S, dP: 64 keys, both K-major
      constexpr uint32_t idesc_q = idesc_bf16(128, D, false, true);        // dQ: A = dS in TMEM, B = K MN-major
      constexpr uint64_t kUnitDesc = (uint64_t)(C::kUnitBytes >> 4);
      const uint64_t dq0 = sdesc_sw128(smem_addr(smem + C::kQOff), 16, 1024);
      const uint64_t ddo0 = sdesc_sw128(smem_addr(smem + C::kDOOff), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_addr(smem + C::kKOff), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_addr(smem + C::kVOff), 16, 1024);
      const uint64_t dkmn0 = sdesc_sw128(smem_addr(smem + C::kKOff), kUnitBox, 1024);
      // S(u) = Q K_u^T into warpgroup u % 2's S columns; dP(u) = dO V_u^T into its dP columns.
      // A operand (Q / dO): 128-row boxes, 16 KB apart; B operand (K / V unit): 64-row boxes, 8 KB apart.
      auto issue_s = [=](int u) {
        const uint64_t bk = dk0 + (uint64_t)(u % ST) * kUnitDesc;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t offa = (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
          const uint64_t offb = (uint64_t)(((kk >> 2) * kUnitBox + (kk & 3) * 32) >> 4);
          umma_ss(tbase + 128u * (u & 1), dq0 + offa, bk + offb, idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars->s_full[u & 1]);
      };
      auto issue_dp = [=](int u) {
        const uint64_t bv = dv0 + (uint64_t)(u % ST) * kUnitDesc;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t offa = (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
          const uint64_t offb = (uint64_t)(((kk >> 2) * kUnitBox + (kk & 3) * 32) >> 4);
          umma_ss(tbase + 128u * (u & 1) + 64u, ddo0 + offa, bv + offb, idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars->dp_full[u & 1]);
      };
      // dQ += dS(u) K_u: 64 keys, 16 per MMA (16 K rows = 2 KB down the unit's boxes).
      auto issue_dq = [=](int u) {
        const uint64_t bk = dkmn0 + (uint64_t)(u % ST) * kUnitDesc;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ts(tbase + C::kDQCol, tbase + 128u * (u & 1) + (uint32_t)kk * 8u, bk + (uint64_t)((kk * 2048) >> 4),
                  idesc_q, (u > 0 || kk > 0) ? 1u : 0u);
      };
      // S and dP of unit u once its K and V have landed.
      auto issue_sdp = [&](int u) {
        if (!mbar_wait(&bars->k_full[u % ST], (u / ST) & 1, wg)) return false;
        tc_fence_after();
        issue_s(u);
        if (!mbar_wait(&bars->v_full[u % ST], (u / ST) & 1, wg)) return false;
        tc_fence_after();
        issue_dp(u);
        return true;
      };
      bool ok = mbar_wait(&bars->qdo_full, 0, wg);
      if (ok) tc_fence_after();
      for (int u = 0; ok && u < 2 && u < n_units; ++u) ok = issue_sdp(u);
      for (int u = 0; ok && u < n_units; ++u) {
        if (!(ok = mbar_wait(&bars->ds_full[u & 1], (u >> 1) & 1, wg))) break;
        tc_fence_after();
        issue_dq(u);
        umma_commit(&bars->kv_empty[u % ST]);  // K_u, V_u: every MMA reading them has been issued
        // S(u+2) overwrites dS(u), which dQ(u) just read: the MMA pipe runs in issue order.
        if (u + 2 < n_units) ok = issue_sdp(u + 2);
      }
      umma_commit(&bars->dq_done);
      umma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ element-wise warps 0..7
    const int hh = warp >> 2;  // this warpgroup takes units hh, hh + 2, ...
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tmem = tbase + lane_off + 128u * hh;
    const uint32_t dp_tmem = s_tmem + 64u;
    const int qrow = qt * kTile + row;
    const size_t ridx = (size_t)bh * p.S_pad + qrow;  // rows past S: LSE2 = +inf, so P = 0
    const float neg_lse2 = -p.lse2[ridx];
    const float dval = p.dvec[ridx];
    const float c = p.scale_log2;
    bool ok = true;
    for (int u = hh, it = 0; u < n_units; u += 2, ++it) {
      const int kv0 = u * kUnit;
      // last visible key of this row within the unit (causal diagonal, or keys past S)
      int last = kUnit - 1;
      if (p.causal) last = min(last, qrow - kv0);
      if (kv0 + kUnit > p.S) last = min(last, p.S - 1 - kv0);
      const bool masked = last < kUnit - 1;

      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[hh], it & 1, wg));
      if (!ok) break;
      tc_fence_after();
      float P[64];
      {
        uint32_t r[64];
        tmem_ld_32x32b_x32(s_tmem, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld_32x32b_x32(s_tmem + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        if (masked) {
#pragma unroll
          for (int x = 0; x < 64; ++x) {
            const float e = ex2_approx(fmaf(__uint_as_float(r[x]), c, neg_lse2));
            P[x] = (x <= last) ? e : 0.f;
          }
        } else {
#pragma unroll
          for (int x = 0; x < 64; ++x) P[x] = ex2_approx(fmaf(__uint_as_float(r[x]), c, neg_lse2));
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->dp_full[hh], it & 1, wg));
      if (!ok) break;
      tc_fence_after();
      uint32_t pk[32];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t d[32];
        tmem_ld_32x32b_x32(dp_tmem + q * 32, d);
        tmem_wait_ld_x32(d);
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int c0 = q * 32 + 2 * x;
          pk[q * 16 + x] = pack_bf16(P[c0] * (__uint_as_float(d[2 * x]) - dval),
                                     P[c0 + 1] * (__uint_as_float(d[2 * x + 1]) - dval));
        }
      }
      tmem_st_32x32b_x32(s_tmem, pk);  // dS, packed bf16, over the first 32 columns of S
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&bars->ds_full[hh]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->dq_done, 0, wg));
    if (ok) {
      tc_fence_after();
      // Warp w stores rows of its lane quarter, columns [hh * D/2, hh * D/2 + D/2).
      uint8_t* stage = smem + C::kQOff;  // Q is no longer read by any MMA
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col0 = hh * (D / 2) + cc * 32;
        uint32_t o[32];
        tmem_ld_32x32b_x32(tbase + lane_off + C::kDQCol + col0, o);
        tmem_wait_ld_x32(o);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(o[8 * u + 0]) * p.scale, __uint_as_float(o[8 * u + 1]) * p.scale);
          w.y = pack_bf16(__uint_as_float(o[8 * u + 2]) * p.scale, __uint_as_float(o[8 * u + 3]) * p.scale);
          w.z = pack_bf16(__uint_as_float(o[8 * u + 4]) * p.scale, __uint_as_float(o[8 * u + 5]) * p.scale);
          w.w = pack_bf16(__uint_as_float(o[8 * u + 6]) * p.scale, __uint_as_float(o[8 * u + 7]) * p.scale);
          const int col = col0 + u * 8;
          const int unit = (col & 63) >> 3;
          *reinterpret_cast<uint4*>(stage + (col >> 6) * kBoxBytes + row * 128 + ((unit ^ (row & 7)) << 4)) = w;
        }
      }
      fence_proxy_async_smem();
      uint32_t phase = 0;
      ok = wg_barrier(&bars->epi_bar, phase, wg);
      if (ok && tid == 0) {
        for (int cb = 0; cb < C::kChunks; ++cb) tma_store_3d(&map_dq, stage + cb * kBoxBytes, cb * kChunk, qt * kTile, bh);
        bulk_commit_group();
        bulk_wait_group_read<0>();
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_bwd_dq_d(const BwdArgs& a, cudaStream_t stream) {
  using C = DqCfg<D>;
  const int n_tiles = ceil_div(a.S, kTile);
  DqKParams p;
  p.lse2 = a.lse2;
  p.dvec = a.dvec;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.S = a.S;
  p.S_pad = n_tiles * kTile;
  p.causal = a.causal;
  p.scale = a.scale;
  p.scale_log2 = a.scale_log2;
  p.status = a.status;
  cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(a.B * a.Hq), (unsigned)n_tiles);
  trace_begin(kKernelBwdDq, stream);
  bwd_dq_kernel<D><<<grid, C::kThreads, C::kSmemBytes, stream>>>(*a.map_q, *a.map_k64, *a.map_v64, *a.map_do,
                                                                 *a.map_dq, p);
  e = cudaGetLastError();
  trace_end(kKernelBwdDq, stream);
  return e;
}

}  // namespace

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream) {
  if (a.D == 64) return launch_bwd_dq_d<64>(a, stream);
  return launch_bwd_dq_d<128>(a, stream);
}

}  // namespace gqa
