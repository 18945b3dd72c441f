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
// One CTA = one (batch, query head, 128-row query tile). Keys stream in
// 128-row units u (keys 128u .. 128u+127), so that every contraction is a
// full-rate 128 x N x 16 MMA. Q and dO are copied once into TMEM, so that all
// three contractions take their A operand from TMEM: the tensor core reads
// only K or V from shared memory (which leaves shared-memory bandwidth to the
// TMA copies), and shared memory holds nothing but the K and V rings.
// Unit u is worked on by element-wise warpgroup u % 2 in TMEM region u % R
// (128 columns; R = 2 at D = 128, 3 at D = 64): S(u) lands there; the
// warpgroup turns it into P (bf16, kept in registers) and releases the
// region; dP(u) is written over it; the warpgroup forms dS = P (dP - D), packs
// it to bf16 over the region's first 64 columns; dQ(u) reads it from there.
// The MMA thread does not follow a fixed order: it polls which of dP, dQ and S
// of the oldest pending units is ready and issues the first that is (dP before
// dQ before S), so that no warpgroup's wait is queued behind an MMA that could
// not start.
// Warp roles (320 threads):
//   warps 0..3  element-wise, even units: thread r owns query row r (TMEM lane r);
//   warps 4..7  element-wise, odd units;
//   warp 8      TMA producer: Q and dO once, then K and V units into two rings;
//   warp 9      MMA issuer (one thread) and TMEM owner.
// TMEM columns: regions [0, 128R); dQ [128R, 128R+D); Q (bf16 pairs)
// [128R+D, 128R+3D/2); dO [128R+3D/2, 128R+2D) -- 512 in all at D = 128 and 64.
// Q and dO arrive by TMA in the last stage of the K and V rings, which the
// ring takes over once they are in TMEM. A unit's K stays resident from S(u)
// to dQ(u), its V from dP(u) only: the K ring has more stages than the V ring.
// Epilogue: dQ * scale in bf16 into the (no longer used) first K stage in the
// TMA box layout, stored by TMA; rows past S are clipped.
#include "common.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kUnit = kTile;  // keys per unit (128)
constexpr int kMaxRegions = 3;

template <int D>
struct DqCfg {
  static constexpr int kChunks = D / kChunk;
  static constexpr int kTileBytes = kTile * D * 2;  // a Q or dO tile, a K or V unit
  static constexpr int kRegions = (D == 64) ? 3 : 2;
  static constexpr int kKStages = (D == 64) ? 8 : 4;
  static constexpr int kVStages = (D == 64) ? 5 : 3;
  static constexpr int kKOff = 0;  // K ring (its first stage: the dQ staging at the end)
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kQStage = kKOff + (kKStages - 1) * kTileBytes;   // Q lands here first
  static constexpr int kDOStage = kVOff + (kVStages - 1) * kTileBytes;  // dO lands here first
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;  // barriers + alignment slack
  static constexpr int kThreads = 320;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kDQCol = kRegions * 128;
  static constexpr uint32_t kQCol = kDQCol + D;
  static constexpr uint32_t kDOCol = kQCol + D / 2;
  static_assert(kDOCol + D / 2 <= kTmemCols, "dQ kernel TMEM columns");
};

template <int KS, int VS>
struct DqBars {
  uint64_t qdo_full;  // Q and dO in shared memory (TMA)
  uint64_t qdo_tmem;  // Q and dO copied into TMEM (8 warp arrivals)
  uint64_t k_full[KS];
  uint64_t k_empty[KS];
  uint64_t v_full[VS];
  uint64_t v_empty[VS];
  uint64_t s_full[kMaxRegions];   // S(u) in region u % R (MMA commit)
  uint64_t s_free[kMaxRegions];   // S(u) read into registers (4 warp arrivals)
  uint64_t dp_full[kMaxRegions];  // dP(u) over it (MMA commit)
  uint64_t ds_full[kMaxRegions];  // dS(u) packed over it (4 warp arrivals)
  uint64_t dq_done;
  uint64_t drain;
  uint64_t epi_bar;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
using DqBarsOf = DqBars<DqCfg<D>::kKStages, DqCfg<D>::kVStages>;

static_assert(sizeof(DqBarsOf<64>) <= DqCfg<64>::kBarBytes && sizeof(DqBarsOf<128>) <= DqCfg<128>::kBarBytes,
              "dQ kernel barriers exceed the bytes reserved for them");
static_assert(DqCfg<64>::kSmemBytes <= 232448 && DqCfg<128>::kSmemBytes <= 232448, "dQ kernel smem over the limit");

struct DqKParams {
  const float* nlse2;  // f32 [B*Hq, S_pad]: -LSE * log2(e), -inf past S
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


__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int D>
__global__ void __launch_bounds__(320, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                  const __grid_constant__ CUtensorMap map_dq, const DqKParams p) {
  using C = DqCfg<D>;
  constexpr int KS = C::kKStages;
  constexpr int VS = C::kVStages;
  constexpr int R = C::kRegions;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  auto* bars = reinterpret_cast<DqBarsOf<D>*>(smem + C::kBarOff);
  griddep_wait();  // the D / -LSE2 rows come from the prep kernel, two launches ahead
  griddep_launch_dependents();

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int bh = blockIdx.x;                            // b * Hq + h
  const int qt = (int)gridDim.y - 1 - (int)blockIdx.y;  // longest query tiles first
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int kvh = b * p.Hkv + h / (p.Hq / p.Hkv);
  // key units this query tile visits: causal, keys up to the tile's last row; else all S keys
  const int n_units = p.causal ? qt + 1 : (p.S + kUnit - 1) / kUnit;
  const WaitGuard wg{&bars->abort_flag, p.status, kWaitLimitNs};
  const int heads_q = (int)gridDim.x;                     // extents for the debug build's checks
  const int heads_kv = heads_q / (p.Hq / p.Hkv);

  if (tid == 0) {
    mbar_init(&bars->qdo_full, 1);
    mbar_init(&bars->qdo_tmem, 8);
    for (int s = 0; s < KS; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int i = 0; i < R; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 4);  // one arrival per warp of the unit's warpgroup
      mbar_init(&bars->dp_full[i], 1);
      mbar_init(&bars->ds_full[i], 4);
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
        const bool q_ok = dbg_tile(c * kChunk, qt * kTile, bh, D, kChunk, 0, p.S, heads_q, p.status);
        tma_load_3d_chk(smem + C::kQStage + c * kBoxBytes, &map_q, &bars->qdo_full, c * kChunk, qt * kTile, bh, q_ok);
        tma_load_3d_chk(smem + C::kDOStage + c * kBoxBytes, &map_do, &bars->qdo_full, c * kChunk, qt * kTile, bh,
                        q_ok);
      }
      // K(u) may reuse its stage once dQ(u - KS) has run, V(u) once dP(u - VS) has; the
      // last stage of each ring is first taken once Q and dO have been copied out of it.
      int k_issued = 0, v_issued = 0;
      for (int u = 0; u < n_units; ++u) {
        const int ks = u % KS;
        if (u >= KS && !mbar_wait(&bars->k_empty[ks], ((u / KS) - 1) & 1, wg)) break;
        if (u == KS - 1 && !mbar_wait(&bars->qdo_tmem, 0, wg)) break;
        mbar_arrive_expect_tx(&bars->k_full[ks], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d_chk(smem + C::kKOff + ks * C::kTileBytes + c * kBoxBytes, &map_k, &bars->k_full[ks],
                          c * kChunk, u * kUnit, kvh,
                          dbg_tile(c * kChunk, u * kUnit, kvh, D, kChunk, 0, p.S, heads_kv, p.status));
        k_issued = u + 1;
        const int vs = u % VS;
        if (u >= VS && !mbar_wait(&bars->v_empty[vs], ((u / VS) - 1) & 1, wg)) break;
        if (u == VS - 1 && !mbar_wait(&bars->qdo_tmem, 0, wg)) break;
        mbar_arrive_expect_tx(&bars->v_full[vs], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d_chk(smem + C::kVOff + vs * C::kTileBytes + c * kBoxBytes, &map_v, &bars->v_full[vs],
                          c * kChunk, u * kUnit, kvh,
                          dbg_tile(c * kChunk, u * kUnit, kvh, D, kChunk, 0, p.S, heads_kv, p.status));
        v_issued = u + 1;
      }
      if (bars->abort_flag) {
        // Let every copy already issued land before the CTA's shared memory goes away.
        mbar_wait_drain(&bars->qdo_full, 0, kWaitLimitNs);
        for (int u = (k_issued > KS ? k_issued - KS : 0); u < k_issued; ++u)
          mbar_wait_drain(&bars->k_full[u % KS], (u / KS) & 1, kWaitLimitNs);
        for (int u = (v_issued > VS ? v_issued - VS : 0); u < v_issued; ++u)
          mbar_wait_drain(&bars->v_full[u % VS], (u / VS) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, kUnit, false, false);  // S, dP: A in TMEM, B K-major
      constexpr uint32_t idesc_q = idesc_bf16(128, D, false, true);        // dQ: A = dS in TMEM, B = K MN-major
      constexpr uint64_t kStageDesc = (uint64_t)(C::kTileBytes >> 4);
      const uint64_t dk0 = sdesc_sw128(smem_addr(smem + C::kKOff), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_addr(smem + C::kVOff), 16, 1024);
      const uint64_t dkmn0 = sdesc_sw128(smem_addr(smem + C::kKOff), kBoxBytes, 1024);
      // S(u) = Q K_u^T and dP(u) = dO V_u^T into region u % R. A: 16 columns of Q (dO) per
      // MMA, 8 TMEM columns of bf16 pairs; B: 128-row boxes of 64 columns, 16 KB apart.
      auto issue_s = [=](int u) {
        const uint32_t dst = tbase + 128u * (uint32_t)(u % R);
        const uint64_t bk = dk0 + (uint64_t)(u % KS) * kStageDesc;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
          umma_ts(dst, tbase + C::kQCol + (uint32_t)kk * 8u, bk + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars->s_full[u % R]);
      };
      auto issue_dp = [=](int u) {
        const uint32_t dst = tbase + 128u * (uint32_t)(u % R);
        const uint64_t bv = dv0 + (uint64_t)(u % VS) * kStageDesc;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
          umma_ts(dst, tbase + C::kDOCol + (uint32_t)kk * 8u, bv + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars->dp_full[u % R]);
        umma_commit(&bars->v_empty[u % VS]);  // V(u): its only MMA has been issued
      };
      // dQ += dS(u) K_u: 128 keys, 16 per MMA (16 K rows = 2 KB down the unit's boxes).
      auto issue_dq = [=](int u) {
        const uint32_t src = tbase + 128u * (uint32_t)(u % R);
        const uint64_t bk = dkmn0 + (uint64_t)(u % KS) * kStageDesc;
#pragma unroll
        for (int kk = 0; kk < kUnit / 16; ++kk)
          umma_ts(tbase + C::kDQCol, src + (uint32_t)kk * 8u, bk + (uint64_t)((kk * 2048) >> 4), idesc_q,
                  (u > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars->k_empty[u % KS]);  // K(u): every MMA reading it has been issued
      };
      // ns, np, nq: the next unit whose S, dP, dQ is to be issued (nq <= np <= ns).
      // S(u) overwrites region u % R, last read by dQ(u - R): issued before it, and the
      // MMA pipe runs in issue order. Every barrier polled here is at most one phase
      // ahead of the last one this thread saw complete, so parity identifies the phase.
      int ns = 0, np = 0, nq = 0;
      bool ok = mbar_wait(&bars->qdo_tmem, 0, wg);
      if (ok) tc_fence_after();
      uint64_t t_last = globaltimer_ns();
      uint32_t idle = 0;
      while (ok && nq < n_units) {
        bool issued = false;
        if (np < ns && mbar_test_wait(&bars->s_free[np % R], (np / R) & 1) &&
            mbar_test_wait(&bars->v_full[np % VS], (np / VS) & 1)) {
          tc_fence_after();
          issue_dp(np++);
          issued = true;
        } else if (nq < np && mbar_test_wait(&bars->ds_full[nq % R], (nq / R) & 1)) {
          tc_fence_after();
          issue_dq(nq++);
          issued = true;
        } else if (ns < n_units && ns - nq < R &&
                   mbar_test_wait(&bars->k_full[ns % KS], (ns / KS) & 1)) {
          tc_fence_after();
          issue_s(ns++);
          issued = true;
        }
        if (issued) {
          idle = 0;
        } else if ((++idle & 15u) == 0) {
          if (idle == 16u) t_last = globaltimer_ns();
          if (*wg.abort_flag) {
            ok = false;
          } else if (globaltimer_ns() - t_last > kWaitLimitNs) {
            *wg.abort_flag = 1;
            atomicOr(p.status, STATUS_TIMEOUT);
            ok = false;
          }
        }
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
    const int qrow = qt * kTile + row;
    const size_t ridx = (size_t)bh * p.S_pad + qrow;  // rows past S: LSE2 = +inf, so P = 0
    const bool r_ok = dbg_range((long long)ridx, 1, (long long)heads_q * p.S_pad, p.status);
    const float neg_lse2 = r_ok ? p.nlse2[ridx] : 0.f;
    const float dval = r_ok ? p.dvec[ridx] : 0.f;
    const float c = p.scale_log2;
    // Q (warpgroup 0) or dO (warpgroup 1) into TMEM: thread r copies row r out of the
    // 128B-swizzled boxes as bf16 pairs, the layout of an MMA A operand in TMEM.
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->qdo_full, 0, wg));
    if (ok) {
      const uint8_t* src = smem + (hh == 0 ? C::kQStage : C::kDOStage);
      const uint32_t dst = tbase + lane_off + (hh == 0 ? C::kQCol : C::kDOCol);
#pragma unroll
      for (int cb = 0; cb < C::kChunks; ++cb) {
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 x = *reinterpret_cast<const uint4*>(src + cb * kBoxBytes + row * 128 + ((j ^ (row & 7)) << 4));
          w[4 * j] = x.x;
          w[4 * j + 1] = x.y;
          w[4 * j + 2] = x.z;
          w[4 * j + 3] = x.w;
        }
        tmem_st_32x32b_x32(dst + 32u * (uint32_t)cb, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&bars->qdo_tmem);  // the MMA may read them; the ring may reuse the stages
    }
    for (int u = hh; ok && u < n_units; u += 2) {
      const int rg = u % R;
      const uint32_t ph = (uint32_t)(u / R) & 1u;
      const uint32_t reg_tmem = tbase + lane_off + 128u * (uint32_t)rg;
      const int kv0 = u * kUnit;
      // last visible key of this row within the unit (causal diagonal, or keys past S)
      int last = kUnit - 1;
      if (p.causal) last = min(last, qrow - kv0);
      if (kv0 + kUnit > p.S) last = min(last, p.S - 1 - kv0);
      const bool masked = last < kUnit - 1;

      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[rg], ph, wg));
      if (!ok) break;
      tc_fence_after();
      // P = exp2(S c - LSE2), packed to bf16 pairs: pp[x] holds keys 2x, 2x + 1.
      uint32_t pp[kUnit / 2];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t r[64];
        tmem_ld_32x32b_x32(reg_tmem + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld_32x32b_x32(reg_tmem + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        if (masked) {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int k0 = 64 * half + 2 * x;
            const float e0 = ex2_approx(fmaf(__uint_as_float(r[2 * x]), c, neg_lse2));
            const float e1 = ex2_approx(fmaf(__uint_as_float(r[2 * x + 1]), c, neg_lse2));
            pp[32 * half + x] = pack_bf16(k0 <= last ? e0 : 0.f, k0 + 1 <= last ? e1 : 0.f);
          }
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x)
            pp[32 * half + x] = pack_bf16(ex2_approx(fmaf(__uint_as_float(r[2 * x]), c, neg_lse2)),
                                          ex2_approx(fmaf(__uint_as_float(r[2 * x + 1]), c, neg_lse2)));
        }
      }
      tc_fence_before();
      mbar_arrive_warp(&bars->s_free[rg]);  // the region may now take dP(u)

      ok = __all_sync(0xffffffffu, mbar_wait(&bars->dp_full[rg], ph, wg));
      if (!ok) break;
      tc_fence_after();
      // dS = P (dP - D), packed: keys 64 half .. 64 half + 63 go to columns 32 half .. 32 half + 31,
      // which hold dP columns that have already been read.
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t d[64];
        tmem_ld_32x32b_x32(reg_tmem + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&d[0]));
        tmem_ld_32x32b_x32(reg_tmem + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&d[32]));
        tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&d[0]));
        tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&d[32]));
        uint32_t pk[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const uint32_t w = pp[32 * half + x];
          pk[x] = pack_bf16(bf16_lo(w) * (__uint_as_float(d[2 * x]) - dval),
                            bf16_hi(w) * (__uint_as_float(d[2 * x + 1]) - dval));
        }
        tmem_st_32x32b_x32(reg_tmem + 32 * half, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&bars->ds_full[rg]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->dq_done, 0, wg));
    if (ok) {
      tc_fence_after();
      // Warp w stores rows of its lane quarter, columns [hh * D/2, hh * D/2 + D/2).
      uint8_t* stage = smem + C::kKOff;  // no MMA reads the K ring any more
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
        for (int cb = 0; cb < C::kChunks; ++cb)
          if (dbg_tile(cb * kChunk, qt * kTile, bh, D, kChunk, 0, p.S, heads_q, p.status))
            tma_store_3d(&map_dq, stage + cb * kBoxBytes, cb * kChunk, qt * kTile, bh);
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
  p.nlse2 = a.nlse2;
  p.dvec = a.dvec;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.S = a.S;
  p.S_pad = n_tiles * kTile;
  p.causal = a.causal;
  p.scale = a.scale;
  p.scale_log2 = a.scale_log2;
  p.status = a.status;
  cudaError_t e = kernel_setup(reinterpret_cast<const void*>(bwd_dq_kernel<D>), C::kSmemBytes, C::kThreads, 0);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(a.B * a.Hq), (unsigned)n_tiles);
  trace_begin(kKernelBwdDq, stream);
  e = launch_pdl(bwd_dq_kernel<D>, grid, dim3(C::kThreads), C::kSmemBytes, stream, *a.map_q, *a.map_k, *a.map_v,
                 *a.map_do, *a.map_dq, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  trace_end(kKernelBwdDq, stream);
  return e;
}

}  // namespace

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream) {
  if (a.D == 64) return launch_bwd_dq_d<64>(a, stream);
  return launch_bwd_dq_d<128>(a, stream);
}

}  // namespace gqa
