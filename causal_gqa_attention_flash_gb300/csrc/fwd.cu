// Forward of fused causal grouped-query attention on sm_103a.
//
// Computes O = softmax(scale * Q K^T + causal mask) V and the per-row
// log-sum-exp with the streaming form the tang page derives ("How tang works",
// section 3, equations (5)-(6)): for each query row three running values --
// the reference max m, the sum l and the accumulator O -- are updated key tile
// by key tile, so that no score ever reaches global memory. Because the combine
// is associative the key loop tiles (section 3, last paragraph); here the tile
// is 128 keys, one tcgen05 M=128 x N=128 MMA.
//
// One CTA = one (batch, query head, 128-row query tile). Warp roles:
//   warp 4      TMA producer: Q once, then K_j / V_j into a ring of stages;
//   warp 5      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               buffers, then O += P_j V_j with P_j read from TMEM;
//   warps 0..3  softmax: thread r owns query row r (TMEM lane r); reads S_j,
//               updates (m, l), writes P_j = exp2(S_j*c - m) as bf16 back into
//               the S_j buffer, rescales O in TMEM when m moves, and finally
//               writes O / l and LSE.
// TMEM columns: S buffer 0 at [0,128), S buffer 1 at [128,256), O at [256,256+D).
// The reference max is only moved when the tile max exceeds it by more than
// 2^8 (lazy rescale); any reference >= the true max gives the same O / l and
// LSE, which is the monoid's regrouping property.
#include "common.h"
#include "ptx.cuh"

namespace gqa {
namespace {

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / kChunk;
  static constexpr int kTileBytes = kTile * D * 2;  // one 128-row bf16 tile of Q, K or V
  static constexpr int kStages = (D == 64) ? 3 : 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers + alignment slack
  static constexpr int kThreads = 192;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 256;
};

template <int ST>
struct FwdBars {
  uint64_t q_full;
  uint64_t k_full[ST];
  uint64_t v_full[ST];
  uint64_t kv_empty[ST];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdKParams {
  uint16_t* o;
  float* lse;
  int Hq, Hkv, S, causal, n_tiles;
  float scale_log2;
  int* status;
};

// Time-bounded wait that ignores the abort flag: used when tearing down after
// an abort, to let copies and MMAs already in flight land before the CTA exits.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

template <int D>
__global__ void __launch_bounds__(192, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const FwdKParams p) {
  using C = FwdCfg<D>;
  constexpr int ST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  auto* bars = reinterpret_cast<FwdBars<ST>*>(smem + C::kBarOff);
  uint8_t* sQ = smem + C::kQOff;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int bh = blockIdx.x;                      // b * Hq + h
  const int qt = (int)gridDim.y - 1 - (int)blockIdx.y;  // longest (most key tiles) first
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int kvh = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int q0 = qt * kTile;
  const int n_kv = p.causal ? (qt + 1) : p.n_tiles;
  const WaitGuard wg{&bars->abort_flag, p.status, kWaitLimitNs};

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 128);
    }
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      mbar_arrive_expect_tx(&bars->q_full, C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_3d(sQ + c * kBoxBytes, &map_q, &bars->q_full, c * kChunk, q0, bh);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % ST;
        const int use = j / ST;
        if (use > 0 && !mbar_wait(&bars->kv_empty[st], (use - 1) & 1, wg)) break;
        uint8_t* sK = smem + C::kKOff + st * C::kTileBytes;
        uint8_t* sV = smem + C::kVOff + st * C::kTileBytes;
        mbar_arrive_expect_tx(&bars->k_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sK + c * kBoxBytes, &map_k, &bars->k_full[st], c * kChunk, j * kTile, kvh);
        mbar_arrive_expect_tx(&bars->v_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sV + c * kBoxBytes, &map_v, &bars->v_full[st], c * kChunk, j * kTile, kvh);
        issued = j + 1;
      }
      if (bars->abort_flag) {
        // Let every copy already issued land before the CTA's shared memory goes away.
        mbar_wait_drain(&bars->q_full, 0, kWaitLimitNs);
        for (int j = (issued > ST ? issued - ST : 0); j < issued; ++j) {
          mbar_wait_drain(&bars->k_full[j % ST], (j / ST) & 1, kWaitLimitNs);
          mbar_wait_drain(&bars->v_full[j % ST], (j / ST) & 1, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, D, false, true);
      const uint32_t o_tmem = tbase + C::kOCol;
      const uint32_t q_addr = smem_addr(sQ);
      auto issue_s = [&](int j) {
        const uint32_t k_addr = smem_addr(smem + C::kKOff + (j % ST) * C::kTileBytes);
        const uint32_t d_tmem = tbase + (uint32_t)(j & 1) * 128u;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * kBoxBytes + (uint32_t)(kk & 3) * 32u;
          umma_ss(d_tmem, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024), idesc_s,
                  kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars->s_full[j & 1]);
      };
      bool ok = mbar_wait(&bars->q_full, 0, wg) && mbar_wait(&bars->k_full[0], 0, wg);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          const int j1 = j + 1;
          if (!(ok = mbar_wait(&bars->k_full[j1 % ST], (j1 / ST) & 1, wg))) break;
          tc_fence_after();
          issue_s(j1);
        }
        if (!(ok = mbar_wait(&bars->p_full[j & 1], (j >> 1) & 1, wg))) break;
        const int st = j % ST;
        if (!(ok = mbar_wait(&bars->v_full[st], (j / ST) & 1, wg))) break;
        tc_fence_after();
        const uint32_t v_addr = smem_addr(smem + C::kVOff + st * C::kTileBytes);
        const uint32_t p_tmem = tbase + (uint32_t)(j & 1) * 128u;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          umma_ts(o_tmem, p_tmem + (uint32_t)kk * 8u, sdesc_sw128(v_addr + (uint32_t)kk * 2048u, kBoxBytes, 1024),
                  idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars->o_done);
        umma_commit(&bars->kv_empty[st]);
      }
      // Every MMA issued completes before TMEM is released.
      umma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0..3)
    const int row = tid;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t o_tmem = tbase + lane_off + C::kOCol;
    const float c = p.scale_log2;
    float m_ref = 0.f, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int buf = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[buf], (j >> 1) & 1, wg));
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_tmem = tbase + lane_off + (uint32_t)buf * 128u;
      uint32_t r[128];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        tmem_ld_32x32b_x32(s_tmem + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * q]));
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&r[32 * q]));

      const int kv0 = j * kTile;
      const bool diag = p.causal && (j == qt);
      const bool tail = !p.causal && (kv0 + kTile > p.S);
      const int last = diag ? row : (tail ? (p.S - kv0 - 1) : (kTile - 1));  // last visible local key
      float s[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(r[i]);
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
      if (diag || tail) {
#pragma unroll
        for (int i = 0; i < 128; i += 4) {
          mx0 = fmaxf(mx0, i + 0 <= last ? s[i + 0] : -INFINITY);
          mx1 = fmaxf(mx1, i + 1 <= last ? s[i + 1] : -INFINITY);
          mx2 = fmaxf(mx2, i + 2 <= last ? s[i + 2] : -INFINITY);
          mx3 = fmaxf(mx3, i + 3 <= last ? s[i + 3] : -INFINITY);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 128; i += 4) {
          mx0 = fmaxf(mx0, s[i + 0]);
          mx1 = fmaxf(mx1, s[i + 1]);
          mx2 = fmaxf(mx2, s[i + 2]);
          mx3 = fmaxf(mx3, s[i + 3]);
        }
      }
      const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
      float alpha = 1.f;
      bool need = false;
      if (j == 0) {
        m_ref = m_tile;
      } else if (m_tile > m_ref + 8.f) {
        alpha = ex2_approx(m_ref - m_tile);
        m_ref = m_tile;
        need = true;
      }
      const float neg_m = -m_ref;
      float sum0 = 0.f, sum1 = 0.f;
      if (diag || tail) {
#pragma unroll
        for (int i = 0; i < 128; i += 2) {
          s[i] = (i <= last) ? ex2_approx(fmaf(s[i], c, neg_m)) : 0.f;
          s[i + 1] = (i + 1 <= last) ? ex2_approx(fmaf(s[i + 1], c, neg_m)) : 0.f;
          sum0 += s[i];
          sum1 += s[i + 1];
        }
      } else {
#pragma unroll
        for (int i = 0; i < 128; i += 2) {
          s[i] = ex2_approx(fmaf(s[i], c, neg_m));
          s[i + 1] = ex2_approx(fmaf(s[i + 1], c, neg_m));
          sum0 += s[i];
          sum1 += s[i + 1];
        }
      }
      l = l * alpha + (sum0 + sum1);

      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O holds the sum up to tile j-1 against the old reference: wait for P_{j-1} V_{j-1}, then rescale.
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done, (j - 1) & 1, wg));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(o_tmem + cc * 32, o);
          tmem_wait_ld_x32(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st_32x32b_x32(o_tmem + cc * 32, o);
        }
      }
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) pk[i] = pack_bf16(s[2 * i], s[2 * i + 1]);
      tmem_st_32x32b_x32(s_tmem + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st_32x32b_x32(s_tmem + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[buf]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done, (n_kv - 1) & 1, wg));
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const int qrow = q0 + row;
      uint16_t* orow = p.o + ((size_t)bh * p.S + qrow) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(o_tmem + cc * 32, o);
        tmem_wait_ld_x32(o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        if (qrow < p.S) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (qrow < p.S) p.lse[(size_t)bh * p.S + qrow] = (m_ref + __log2f(l)) * 0.69314718055994530942f;
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  FwdKParams p;
  p.o = static_cast<uint16_t*>(a.o);
  p.lse = a.lse;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.S = a.S;
  p.causal = a.causal;
  p.n_tiles = ceil_div(a.S, kTile);
  p.scale_log2 = a.scale_log2;
  p.status = a.status;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(a.B * a.Hq), (unsigned)p.n_tiles);
  trace_begin(kKernelFwd, stream);
  fwd_kernel<D><<<grid, C::kThreads, C::kSmemBytes, stream>>>(*a.map_q, *a.map_k, *a.map_v, p);
  e = cudaGetLastError();
  trace_end(kKernelFwd, stream);
  return e;
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.D == 64) return launch_fwd_d<64>(a, stream);
  return launch_fwd_d<128>(a, stream);
}

}  // namespace gqa
