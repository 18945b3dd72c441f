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
// One CTA = one (batch, query head) and two consecutive 128-row query tiles,
// A (rows q0..q0+127) and B (rows q0+128..q0+255), which share every K/V tile
// the TMA brings in. Warp roles (384 threads, three warpgroups):
//   warps 0..3  softmax of tile A: thread r owns row r of A (TMEM lane r);
//   warps 4..7  softmax of tile B (same, lanes 0..127 through the lane quarter w % 4);
//   warp 8      TMA producer: Q_A, Q_B once, then K_j into a ring of stages;
//   warp 9      MMA issuer (one thread) and TMEM owner;
//   warp 10     TMA producer: V_j into a ring of stages; warp 11 idle.
// Registers: launched at kLaunchRegs per thread; the producer warpgroup drops
// to kLowRegs and the two softmax warpgroups rise to kHighRegs (setmaxnreg).
// The MMA thread alternates between the tiles: while softmax A works on S_A(j)
// the tensor core runs P_B(j-1) V_{j-1} and S_B(j); while softmax B works on
// S_B(j) it runs P_A(j) V_j and S_A(j+1). Each softmax reads S, updates
// (m, l), and writes P = exp2(S c - m) as bf16 back into the S columns, where
// the next P V MMA reads it as its A operand.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,256+D), O_B [256+D,256+2D).
// The reference max moves only when a tile max exceeds it by more than 8
// (log2 units): any reference >= the true max gives the same O / l and LSE,
// the regrouping property of the monoid. Because S_X(j) is issued after
// P_X(j-1) V_{j-1} on the same in-order MMA stream, its completion also
// means the previous P V is done, so O can be rescaled right away.
// Epilogue: O / l in bf16 is written into the tile's (no longer needed) Q
// buffer in the TMA box layout and stored by TMA; rows past S are clipped.
// Queries may be fewer than keys (Sq <= Sk, bottom-right causal alignment), and
// a batch may be packed: sequences of different lengths laid end to end along
// the row axis, each CTA reading its sequence's bounds, the last ragged query
// tile of a sequence storing its rows one by one.
#include "common.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace gqa {
namespace {

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / kChunk;
  static constexpr int kTileBytes = kTile * D * 2;  // one 128-row bf16 tile of Q, K, V or O
  // K and V ring depths. V_j is needed one MMA-pair later in the key step than K_j and its stage
  // is released later (after both P V products), so at D = 128 the V ring takes the third stage
  // that 227 KB of shared memory leave room for.
  static constexpr int kKStages = (D == 64) ? 4 : 2;
  static constexpr int kVStages = (D == 64) ? 4 : 3;
  static constexpr int kQOff = 0;                   // Q_A, Q_B (reused as O staging)
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers + alignment slack
  static constexpr int kThreads = 384;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 256;
  static constexpr int kLaunchRegs = 168;  // 65536 / 384, rounded down to a multiple of 8
  static constexpr int kLowRegs = 104;
  static constexpr int kHighRegs = 200;
  static_assert(2 * 128 * kHighRegs + 128 * kLowRegs <= kThreads * kLaunchRegs, "register split exceeds the launch");
};

template <int KST, int VST>
struct FwdBars {
  uint64_t q_full;
  uint64_t k_full[KST];
  uint64_t v_full[VST];
  uint64_t k_empty[KST];
  uint64_t v_empty[VST];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t drain;
  uint64_t wg_bar[2];  // one per softmax warpgroup
  uint64_t q_ready[2]; // rotary embedding: tile X's queries rotated in shared memory
  uint32_t tmem_base;
  int abort_flag;
};

static_assert(sizeof(FwdBars<FwdCfg<64>::kKStages, FwdCfg<64>::kVStages>) <= 256 &&
                  sizeof(FwdBars<FwdCfg<128>::kKStages, FwdCfg<128>::kVStages>) <= 256,
              "forward barriers exceed the 256 bytes reserved for them");
static_assert(FwdCfg<64>::kSmemBytes <= 232448 && FwdCfg<128>::kSmemBytes <= 232448, "forward smem over the limit");

struct FwdKParams {
  float* lse;
  uint16_t* o;         // O itself: packed batches store a sequence's ragged last tile row by row
  const int* cu_q;     // packed batches: sequence bounds [nseq + 1] (nullptr: dense batch)
  const int* cu_k;
  int Tq, Tk;          // packed batches: total query and key rows
  int max_seqlen_q;    // packed batches: bound on any sequence's query rows
  const float* rope_cos;  // rotary tables [S, D/2] (nullptr: none); dense batches only
  const float* rope_sin;
  // Dense batch: Sq query rows against Sk >= Sq keys; query row r sits at absolute position
  // koff + r, koff = Sk - Sq (0 for self-attention), and (causal) sees keys j <= koff + r.
  int Hq, Hkv, Sq, Sk, koff, causal, n_ktiles;
  float scale_log2;
  int* status;
};

// The rows one CTA works on: its sequence's query and key counts and where they start.
struct FwdGeom {
  int Sq, Sk, koff, n_ktiles;
  int q_row0, k_row0;    // first query / key row of the sequence in its tensor map
  int q_coord, kv_coord; // outermost tensor-map coordinate of the query head and of its KV head
  size_t lse_base;       // LSE index of the sequence's first query row
};

// Dense batch: (b, h) = blockIdx.x. Packed batch: sequence blockIdx.x / Hq, head blockIdx.x % Hq,
// bounds read from cu_q / cu_k and checked; returns false (status bit set) for bounds that are
// not a valid packing, and the CTA does nothing.
__device__ __forceinline__ bool fwd_geom(const FwdKParams& p, int bh, FwdGeom& g) {
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int G = p.Hq / p.Hkv;
  if (p.cu_q == nullptr) {
    g.Sq = p.Sq;
    g.Sk = p.Sk;
    g.q_row0 = 0;
    g.k_row0 = 0;
    g.q_coord = bh;
    g.kv_coord = b * p.Hkv + h / G;
    g.lse_base = (size_t)bh * p.Sq;
  } else {
    const int q0 = __ldg(p.cu_q + b), q1 = __ldg(p.cu_q + b + 1);
    const int k0 = __ldg(p.cu_k + b), k1 = __ldg(p.cu_k + b + 1);
    if (q0 < 0 || q1 < q0 || q1 > p.Tq || k0 < 0 || k1 < k0 || k1 > p.Tk || q1 - q0 > k1 - k0 ||
        q1 - q0 > p.max_seqlen_q)
      return false;
    g.Sq = q1 - q0;
    g.Sk = k1 - k0;
    g.q_row0 = q0;
    g.k_row0 = k0;
    g.q_coord = h;
    g.kv_coord = h / G;
    g.lse_base = (size_t)h * p.Tq + q0;
  }
  g.koff = g.Sk - g.Sq;
  g.n_ktiles = (g.Sk + kTile - 1) / kTile;
  return true;
}

// Time-bounded wait that ignores the abort flag: used when tearing down after
// an abort, to let copies and MMAs already in flight land before the CTA exits.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Row max of one 128-key score row held in registers. Masked tiles (the
// causal diagonal, the ragged last tile) exclude keys past `last`; the
// unmasked path (all other tiles) has no per-key select.
template <bool kMasked>
__device__ __forceinline__ float row_max(const uint32_t (&r)[128], int last) {
  float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
  for (int i = 0; i < 128; i += 8) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[k] = __uint_as_float(r[i + k]);
      if (kMasked) v[k] = (i + k <= last) ? v[k] : -INFINITY;
    }
    a0 = fmax3(a0, v[0], v[1]);
    a1 = fmax3(a1, v[2], v[3]);
    a2 = fmax3(a2, v[4], v[5]);
    a3 = fmax3(a3, v[6], v[7]);
  }
  return fmax3(a0, a1, fmaxf(a2, a3));
}

// Masked tiles by 32-column chunks. The visible keys of a row are the prefix [0, last]; lo and hi
// are the smallest and largest `last` of the warp (warp-uniform). A chunk every row of the warp
// sees in full takes the unmasked form, a chunk no row of the warp sees is skipped (its P is 0),
// and only the chunk(s) between take the per-key select: on the causal diagonal one chunk of four.
__device__ __forceinline__ float row_max_chunked(const uint32_t (&r)[128], int last, int lo, int hi) {
  float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (32 * q > hi) continue;
    const bool full = 32 * q + 31 <= lo;
#pragma unroll
    for (int i = 32 * q; i < 32 * q + 32; i += 8) {
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        v[k] = __uint_as_float(r[i + k]);
        if (!full) v[k] = (i + k <= last) ? v[k] : -INFINITY;
      }
      a0 = fmax3(a0, v[0], v[1]);
      a1 = fmax3(a1, v[2], v[3]);
      a2 = fmax3(a2, v[4], v[5]);
      a3 = fmax3(a3, v[6], v[7]);
    }
  }
  return fmax3(a0, a1, fmaxf(a2, a3));
}

// P = exp2(S c - m) for one row, packed to bf16 pairs and stored into the
// row's S columns (32 columns per tcgen05.st); returns the row sum of P. The
// sum runs in eight independent partial sums: the pass is latency-bound, and a
// two-accumulator chain of 64 dependent adds cost 6% of the forward.
template <bool kMasked>
__device__ __forceinline__ float exp_pack_store(const uint32_t (&r)[128], int last, float c, float neg_m,
                                                uint32_t s_tmem) {
  float sm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t pk[16];
#pragma unroll
    for (int x2 = 0; x2 < 16; ++x2) {
      const int i = q * 32 + 2 * x2;
      float e0 = ex2_approx(fmaf(__uint_as_float(r[i]), c, neg_m));
      float e1 = ex2_approx(fmaf(__uint_as_float(r[i + 1]), c, neg_m));
      if (kMasked) {
        e0 = (i <= last) ? e0 : 0.f;
        e1 = (i + 1 <= last) ? e1 : 0.f;
      }
      sm[(x2 & 3) * 2] += e0;
      sm[(x2 & 3) * 2 + 1] += e1;
      pk[x2] = pack_bf16(e0, e1);
    }
    tmem_st_32x32b_x16(s_tmem + q * 16, pk);
  }
  return ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
}

// exp_pack_store for a masked tile, by 32-column chunks as row_max_chunked.
__device__ __forceinline__ float exp_pack_store_chunked(const uint32_t (&r)[128], int last, int lo, int hi, float c,
                                                        float neg_m, uint32_t s_tmem) {
  float sm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t pk[16];
    if (32 * q > hi) {
#pragma unroll
      for (int x2 = 0; x2 < 16; ++x2) pk[x2] = 0u;
    } else {
      const bool full = 32 * q + 31 <= lo;
#pragma unroll
      for (int x2 = 0; x2 < 16; ++x2) {
        const int i = q * 32 + 2 * x2;
        float e0 = ex2_approx(fmaf(__uint_as_float(r[i]), c, neg_m));
        float e1 = ex2_approx(fmaf(__uint_as_float(r[i + 1]), c, neg_m));
        if (!full) {
          e0 = (i <= last) ? e0 : 0.f;
          e1 = (i + 1 <= last) ? e1 : 0.f;
        }
        sm[(x2 & 3) * 2] += e0;
        sm[(x2 & 3) * 2 + 1] += e1;
        pk[x2] = pack_bf16(e0, e1);
      }
    }
    tmem_st_32x32b_x16(s_tmem + q * 16, pk);
  }
  return ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
}

// Number of key tiles query tile qt visits; 0 if the tile lies past Sq.
__device__ __forceinline__ int kv_tiles_of(int qt, const FwdGeom& g, int causal) {
  if (qt * kTile >= g.Sq) return 0;
  if (!causal) return g.n_ktiles;
  const int last_row = min(g.Sq - 1, qt * kTile + kTile - 1);
  return (g.koff + last_row) / kTile + 1;
}

// kRope: queries are turned by the rotary embedding as they land in shared memory.
template <int D, bool kRope>
__global__ void __launch_bounds__(384, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
               const FwdKParams p) {
  using C = FwdCfg<D>;
  constexpr int ST = C::kKStages;   // K ring
  constexpr int VST = C::kVStages;  // V ring
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  auto* bars = reinterpret_cast<FwdBars<ST, VST>*>(smem + C::kBarOff);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int bh = blockIdx.x;                                   // b * Hq + h
  const int pair = (int)gridDim.y - 1 - (int)blockIdx.y;       // longest pairs first
  FwdGeom g;
  if (!fwd_geom(p, bh, g)) {
    if (tid == 0) atomicOr(p.status, STATUS_BAD_SEQLENS);
    return;
  }
  const int qtA = 2 * pair, qtB = 2 * pair + 1;
  const int nA = kv_tiles_of(qtA, g, p.causal);
  const int nB = kv_tiles_of(qtB, g, p.causal);
  const int n_kv = nA > nB ? nA : nB;
  if (nA == 0) return;  // a packed batch's short sequence: no query tile of this CTA exists
  const WaitGuard wg{&bars->abort_flag, p.status, kWaitLimitNs};
  // Extents of the tensors this CTA addresses, for the debug build's coordinate checks: heads of
  // the query / key maps and their rows (a packed CTA stays within its own sequence's rows).
  const int heads_q = p.cu_q ? p.Hq : (int)gridDim.x;
  const int heads_kv = p.cu_q ? p.Hkv : (int)gridDim.x / (p.Hq / p.Hkv);
  const int rows_q = p.cu_q ? p.Tq : p.Sq;

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);  // one arrival per softmax warp
      mbar_init(&bars->o_done[i], 1);
    }
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->wg_bar[0], 4);
    mbar_init(&bars->wg_bar[1], 4);
    mbar_init(&bars->q_ready[0], 4);
    mbar_init(&bars->q_ready[1], 4);
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
  if (warp >= 8) {
   setmaxnreg_dec<C::kLowRegs>();
   if (warp == 8) {
    // ------------------------------------------------------------ TMA producer: Q, then the K ring
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      // Q_B only when tile B has rows (its buffer is otherwise never read)
      const int nq = nB > 0 ? 2 : 1;
      mbar_arrive_expect_tx(&bars->q_full, nq * C::kTileBytes);
      for (int t = 0; t < nq; ++t)
        for (int c = 0; c < C::kChunks; ++c) {
          const int r = g.q_row0 + (qtA + t) * kTile;
          tma_load_3d_chk(smem + C::kQOff + t * C::kTileBytes + c * kBoxBytes, &map_q, &bars->q_full, c * kChunk, r,
                          g.q_coord, dbg_tile(c * kChunk, r, g.q_coord, D, kChunk, g.q_row0, g.q_row0 + g.Sq,
                                              heads_q, p.status));
        }
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % ST;
        const int use = j / ST;
        if (use > 0 && !mbar_wait(&bars->k_empty[st], (use - 1) & 1, wg)) break;
        mbar_arrive_expect_tx(&bars->k_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          const int r = g.k_row0 + j * kTile;
          tma_load_3d_chk(smem + C::kKOff + st * C::kTileBytes + c * kBoxBytes, &map_k, &bars->k_full[st],
                          c * kChunk, r, g.kv_coord,
                          dbg_tile(c * kChunk, r, g.kv_coord, D, kChunk, g.k_row0, g.k_row0 + g.Sk, heads_kv,
                                   p.status));
        }
        issued = j + 1;
      }
      if (bars->abort_flag) {
        // Let every copy already issued land before the CTA's shared memory goes away.
        mbar_wait_drain(&bars->q_full, 0, kWaitLimitNs);
        for (int j = (issued > ST ? issued - ST : 0); j < issued; ++j)
          mbar_wait_drain(&bars->k_full[j % ST], (j / ST) & 1, kWaitLimitNs);
      }
    }
   } else if (warp == 10) {
    // ------------------------------------------------------------ TMA producer: the V ring
    if (lane == 0) {
      tma_prefetch_desc(&map_v);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % VST;
        const int use = j / VST;
        if (use > 0 && !mbar_wait(&bars->v_empty[st], (use - 1) & 1, wg)) break;
        mbar_arrive_expect_tx(&bars->v_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          const int r = g.k_row0 + j * kTile;
          tma_load_3d_chk(smem + C::kVOff + st * C::kTileBytes + c * kBoxBytes, &map_v, &bars->v_full[st],
                          c * kChunk, r, g.kv_coord,
                          dbg_tile(c * kChunk, r, g.kv_coord, D, kChunk, g.k_row0, g.k_row0 + g.Sk, heads_kv,
                                   p.status));
        }
        issued = j + 1;
      }
      if (bars->abort_flag) {
        for (int j = (issued > VST ? issued - VST : 0); j < issued; ++j)
          mbar_wait_drain(&bars->v_full[j % VST], (j / VST) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, D, false, true);
      // S_X(j) = Q_X K_j^T into the S columns of tile X.
      // Descriptors are built once; an MMA only adds a compile-time offset (the start-address field
      // is the low 14 bits of the descriptor and never carries). The issuing thread shares its SMSP
      // with softmax warps, so the fewer instructions per MMA, the closer the tensor core runs to its rate.
      const uint64_t dq0 = sdesc_sw128(smem_addr(smem + C::kQOff), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_addr(smem + C::kKOff), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_addr(smem + C::kVOff), kBoxBytes, 1024);
      constexpr uint64_t kTileDesc = (uint64_t)(C::kTileBytes >> 4);  // descriptor step of one tile
      // S_X(j) = Q_X K_j^T into the S columns of tile X.
      auto issue_s = [=](int x, int j) {
        const uint64_t a = dq0 + (uint64_t)x * kTileDesc;
        const uint64_t bk = dk0 + (uint64_t)(j % ST) * kTileDesc;
        const uint32_t d_tmem = tbase + (uint32_t)x * 128u;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
          umma_ss(d_tmem, a + off, bk + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars->s_full[x]);
      };
      // O_X += P_X(j) V_j, P_X(j) read from the S columns of tile X.
      auto issue_pv = [=](int x, int j) {
        const uint64_t bv = dv0 + (uint64_t)(j % VST) * kTileDesc;
        const uint32_t p_tmem = tbase + (uint32_t)x * 128u;
        const uint32_t o_tmem = tbase + C::kOCol + (uint32_t)x * D;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts(o_tmem, p_tmem + (uint32_t)kk * 8u, bv + (uint64_t)((kk * 2048) >> 4), idesc_o,
                  (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars->o_done[x]);
      };
      // K_j is released once the last S MMA reading it completes, V_j once both P V MMAs do:
      // the K ring refills a full key tile earlier than a shared K/V stage would.
      bool ok = mbar_wait(&bars->q_full, 0, wg) && mbar_wait(&bars->k_full[0], 0, wg);
      if (kRope && ok) {  // the softmax warps rotate their tile's queries first
        ok = (nA == 0 || mbar_wait(&bars->q_ready[0], 0, wg)) && (nB == 0 || mbar_wait(&bars->q_ready[1], 0, wg));
      }
      if (ok) {
        tc_fence_after();
        if (nA > 0) issue_s(0, 0);
        if (nB > 0) issue_s(1, 0);
        umma_commit(&bars->k_empty[0]);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const int vst = j % VST;
        const int j1 = j + 1;
        const int st1 = j1 % ST;
        if (!(ok = mbar_wait(&bars->v_full[vst], (j / VST) & 1, wg))) break;
        if (j < nA) {
          if (!(ok = mbar_wait(&bars->p_full[0], j & 1, wg))) break;
          tc_fence_after();
          issue_pv(0, j);
          if (j1 < nA) {
            if (!(ok = mbar_wait(&bars->k_full[st1], (j1 / ST) & 1, wg))) break;
            tc_fence_after();
            issue_s(0, j1);
          }
        }
        if (j < nB) {
          if (!(ok = mbar_wait(&bars->p_full[1], j & 1, wg))) break;
          tc_fence_after();
          issue_pv(1, j);
          if (j1 < nB) {
            if (!(ok = mbar_wait(&bars->k_full[st1], (j1 / ST) & 1, wg))) break;
            tc_fence_after();
            issue_s(1, j1);
          }
        }
        if (j1 < n_kv) umma_commit(&bars->k_empty[st1]);
        umma_commit(&bars->v_empty[vst]);
      }
      // Every MMA issued completes before TMEM is released.
      umma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, kWaitLimitNs);
    }
   }
  } else {
    // ------------------------------------------------------------ softmax (tile X = warp / 4)
    setmaxnreg_inc<C::kHighRegs>();
    const int x = warp >> 2;
    const int row = tid & 127;
    const int qt = qtA + x;
    const int n_x = x ? nB : nA;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tmem = tbase + lane_off + (uint32_t)x * 128u;
    const uint32_t o_tmem = tbase + lane_off + C::kOCol + (uint32_t)x * D;
    const float c = p.scale_log2;
    float m_ref = 0.f, l = 0.f;
    bool ok = true;
    if (kRope && n_x > 0) {
      // Rotary embedding: each thread turns its own query row of tile X in shared memory
      // (rows past S hold zeros and have no table row).
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full, 0, wg));
      const int qpos = qt * kTile + row;
      if (ok && qpos < g.Sq && dbg_range((long long)qpos * (D / 2), D / 2, (long long)p.Sq * (D / 2), p.status))
        rope_rotate_row_smem<D>(smem + C::kQOff + x * C::kTileBytes, row, p.rope_cos + (size_t)qpos * (D / 2),
                                p.rope_sin + (size_t)qpos * (D / 2), 1.f);
      fence_proxy_async_smem();
      mbar_arrive_warp(&bars->q_ready[x]);
    }
    for (int j = 0; j < n_x; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[x], j & 1, wg));
      if (!ok) break;
      tc_fence_after();
      uint32_t r[128];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        tmem_ld_32x32b_x32(s_tmem + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * q]));
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&r[32 * q]));

      const int kv0 = j * kTile;
      // last visible local key of this row in key tile j: the causal bound koff + q - kv0 and the
      // end of the keys; tiles where some row sees fewer than 128 keys take the masked path.
      const int qpos = g.koff + qt * kTile;  // absolute position of the tile's first row
      const bool diag = p.causal && (qpos < kv0 + kTile - 1);
      const bool tail = kv0 + kTile > g.Sk;
      int last = kTile - 1;
      if (diag) last = min(last, qpos + row - kv0);
      if (tail) last = min(last, g.Sk - kv0 - 1);
      const bool masked = diag || tail;  // uniform over the CTA's tile
      int lo = last, hi = last;
      if (masked) {
        lo = __reduce_min_sync(0xffffffffu, last);
        hi = __reduce_max_sync(0xffffffffu, last);
      }
      const float mx = masked ? row_max_chunked(r, last, lo, hi) : row_max<false>(r, last);
      const float m_tile = mx * c;
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
      const float rsum = masked ? exp_pack_store_chunked(r, last, lo, hi, c, neg_m, s_tmem)
                                : exp_pack_store<false>(r, last, c, neg_m, s_tmem);
      l = l * alpha + rsum;

      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O_X holds the sum up to tile j-1 against the old reference. P_X(j-1) V_{j-1} completed
        // before S_X(j) did (same in-order MMA stream); the wait below returns at once.
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done[x], (j - 1) & 1, wg));
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
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&bars->p_full[x]);
    }
    if (ok && n_x > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done[x], (n_x - 1) & 1, wg));
    if (ok && n_x > 0) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const int qrow = qt * kTile + row;
      // A packed batch's last, ragged query tile must not write the rows past its sequence (they
      // belong to the next one): it stores its rows one by one. Every other tile goes through TMA.
      const bool rowwise = p.cu_q != nullptr && (qt + 1) * kTile > g.Sq;
      uint8_t* stage = smem + C::kQOff + x * C::kTileBytes;  // Q_X is no longer read by any MMA
      uint16_t* orow = p.o + ((size_t)g.q_coord * p.Tq + g.q_row0 + qrow) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(o_tmem + cc * 32, o);
        tmem_wait_ld_x32(o);
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // 16-byte units of 8 columns
          uint4 w;
          w.x = pack_bf16(__uint_as_float(o[8 * u + 0]) * inv_l, __uint_as_float(o[8 * u + 1]) * inv_l);
          w.y = pack_bf16(__uint_as_float(o[8 * u + 2]) * inv_l, __uint_as_float(o[8 * u + 3]) * inv_l);
          w.z = pack_bf16(__uint_as_float(o[8 * u + 4]) * inv_l, __uint_as_float(o[8 * u + 5]) * inv_l);
          w.w = pack_bf16(__uint_as_float(o[8 * u + 6]) * inv_l, __uint_as_float(o[8 * u + 7]) * inv_l);
          const int col = cc * 32 + u * 8;      // first column of the unit
          if (rowwise) {
            if (qrow < g.Sq &&
                dbg_range(((long long)g.q_coord * p.Tq + g.q_row0 + qrow) * D + col, 8, (long long)heads_q * rows_q * D,
                          p.status))
              *reinterpret_cast<uint4*>(orow + col) = w;
          } else {
            const int unit = (col & 63) >> 3;     // unit within the 128-byte row of its box
            *reinterpret_cast<uint4*>(stage + (col >> 6) * kBoxBytes + row * 128 + ((unit ^ (row & 7)) << 4)) = w;
          }
        }
      }
      if (!rowwise) {
        fence_proxy_async_smem();
        uint32_t wg_phase = 0;
        ok = wg_barrier(&bars->wg_bar[x], wg_phase, wg);
        if (ok && row == 0) {
          for (int cb = 0; cb < C::kChunks; ++cb)
            if (dbg_tile(cb * kChunk, g.q_row0 + qt * kTile, g.q_coord, D, kChunk, g.q_row0, g.q_row0 + g.Sq, heads_q,
                         p.status))
              tma_store_3d(&map_o, stage + cb * kBoxBytes, cb * kChunk, g.q_row0 + qt * kTile, g.q_coord);
          bulk_commit_group();
        }
      }
      if (qrow < g.Sq && dbg_range((long long)g.lse_base + qrow, 1, (long long)heads_q * rows_q, p.status))
        p.lse[g.lse_base + qrow] = (m_ref + __log2f(l)) * 0.69314718055994530942f;
      if (!rowwise && row == 0) bulk_wait_group_read<0>();
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
cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  FwdKParams p;
  p.lse = a.lse;
  p.o = static_cast<uint16_t*>(a.o);
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.Tq = a.Sq;
  p.Tk = a.Sk;
  p.max_seqlen_q = a.max_seqlen_q;
  p.rope_cos = a.rope_cos;
  p.rope_sin = a.rope_sin;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.koff = a.Sk - a.Sq;
  p.causal = a.causal;
  p.n_ktiles = ceil_div(a.Sk, kTile);
  p.scale_log2 = a.scale_log2;
  p.status = a.status;
  auto kern = a.rope_cos ? fwd_kernel<D, true> : fwd_kernel<D, false>;
  // The setmaxnreg split must fit the registers the block is launched with, or the
  // increase would wait forever: kernel_setup refuses the launch otherwise.
  cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads,
                               2 * 128 * C::kHighRegs + 128 * C::kLowRegs);
  if (e != cudaSuccess) return e;
  // Packed batch: one row of CTAs per (sequence, head), enough pairs for the longest sequence.
  const int rows = a.cu_q ? a.max_seqlen_q : a.Sq;
  dim3 grid((unsigned)(a.B * a.Hq), (unsigned)ceil_div(rows, 2 * kTile));
  trace_begin(kKernelFwd, stream);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(*a.map_q, *a.map_k, *a.map_v, *a.map_o, p);
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
