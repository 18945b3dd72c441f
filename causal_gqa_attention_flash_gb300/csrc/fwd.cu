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
//   thread 0    (of warp 0) issues Q_A and K_0 right after initialising the barriers;
//   warp 8      TMA producer: Q_B and V_0, then K_j and V_j into their rings of
//               stages, and an L2 prefetch of the query tiles of the CTA one wave later;
//   warp 9      MMA issuer (one thread) and TMEM owner; warps 10, 11 idle.
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
#include <algorithm>
#include <functional>
#include <mutex>
#include <queue>
#include <vector>

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
  uint64_t q_full[2];  // Q_A, Q_B (separate, so that S_A(0) need not wait for Q_B)
  uint64_t kv_full[KST];  // K_j and V_j both landed (indexed by K_j's stage); for j = 0, V_0 only
  uint64_t k0_full;       // K_0, so that the first S products need not wait for V_0
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
  // Key-range split of a dense forward (kcap > 0): the key tiles of tile A of a query-tile pair
  // are cut into ceil(nA / kcap) contiguous parts, one CTA each (the last part also takes tile B's
  // extra key tile); grid y enumerates the (pair, part) pairs, longest pairs first. Each part
  // writes tile A's and tile B's unnormalised O and (m, l) to its slot of `part`, and the combine
  // kernel merges the slots of a pair with the monoid combine.
  int kcap, n_pairs, parts_per_bh;
  float* part;
  // Division-free geometry at the start of every CTA: G = Hq / Hkv, and the multipliers of
  // udiv_by (ceil(2^64 / d), 0 for d = 1) for Hq and G.
  int G;
  unsigned long long div_hq, div_g;
  // SMs of the device: the CTA that will take this CTA's place one wave later is n_sm grid
  // positions further on (one forward CTA per SM); its query tiles are prefetched into L2.
  // 0: no prefetch (queries larger than half the L2, where the prefetched tiles would mostly be
  // evicted before their CTA starts and read from DRAM twice).
  int n_sm;
};

// n / d for 0 <= n < 2^32 and 1 <= d < 2^32, with m = ceil(2^64 / d) (0 for d = 1): the high half
// of n m is exact because n (m - 2^64 / d) < 2^-32 stays below the distance 1/d from n / d to
// the next integer. The integer divide instruction sequence and its constant loads are not
// cheap at the start of a CTA that runs for a few microseconds.
__device__ __forceinline__ int udiv_by(int n, int d, unsigned long long m) {
  return d == 1 ? n : (int)__umul64hi((unsigned long long)(unsigned)n, m);
}
inline unsigned long long udiv_magic(int d) { return d <= 1 ? 0ull : ~0ull / (unsigned long long)d + 1ull; }

}  // namespace

// The device's L2 size in bytes (0 if unknown), looked up once per device (api.cu).
int device_l2_bytes();

namespace {

// Position of grid row y in the split forward: pair, part, parts of the pair, and the index of
// the pair's first slot among its head's slots (only split pairs keep slots).
struct FwdSplitPos {
  int pair, part, parts, pidx;
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
  const int b = udiv_by(bh, p.Hq, p.div_hq);
  const int h = bh - b * p.Hq;
  const int hkv = udiv_by(h, p.G, p.div_g);
  if (p.cu_q == nullptr) {
    g.Sq = p.Sq;
    g.Sk = p.Sk;
    g.q_row0 = 0;
    g.k_row0 = 0;
    g.q_coord = bh;
    g.kv_coord = b * p.Hkv + hkv;
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
    g.kv_coord = hkv;
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
// two-accumulator chain of 64 dependent adds cost 6% of the forward. The
// argument and the sums take the paired f32 instructions (two columns each).
template <bool kMasked>
__device__ __forceinline__ float exp_pack_store(const uint32_t (&r)[128], int last, float c, float neg_m,
                                                uint32_t s_tmem) {
  float2 sm[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  const float2 c2 = make_float2(c, c), nm2 = make_float2(neg_m, neg_m);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t pk[16];
#pragma unroll
    for (int x2 = 0; x2 < 16; ++x2) {
      const int i = q * 32 + 2 * x2;
      const float2 a = ffma2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), c2, nm2);
      float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
      if (kMasked) {
        e.x = (i <= last) ? e.x : 0.f;
        e.y = (i + 1 <= last) ? e.y : 0.f;
      }
      sm[x2 & 3] = fadd2(sm[x2 & 3], e);
      pk[x2] = pack_bf16(e.x, e.y);
    }
    tmem_st_32x32b_x16(s_tmem + q * 16, pk);
  }
  return ((sm[0].x + sm[0].y) + (sm[1].x + sm[1].y)) + ((sm[2].x + sm[2].y) + (sm[3].x + sm[3].y));
}

// exp_pack_store for a masked tile, by 32-column chunks as row_max_chunked.
__device__ __forceinline__ float exp_pack_store_chunked(const uint32_t (&r)[128], int last, int lo, int hi, float c,
                                                        float neg_m, uint32_t s_tmem) {
  float2 sm[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  const float2 c2 = make_float2(c, c), nm2 = make_float2(neg_m, neg_m);
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
        const float2 a = ffma2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), c2, nm2);
        float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
        if (!full) {
          e.x = (i <= last) ? e.x : 0.f;
          e.y = (i + 1 <= last) ? e.y : 0.f;
        }
        sm[x2 & 3] = fadd2(sm[x2 & 3], e);
        pk[x2] = pack_bf16(e.x, e.y);
      }
    }
    tmem_st_32x32b_x16(s_tmem + q * 16, pk);
  }
  return ((sm[0].x + sm[0].y) + (sm[1].x + sm[1].y)) + ((sm[2].x + sm[2].y) + (sm[3].x + sm[3].y));
}

// Number of key tiles query tile qt visits; 0 if the tile lies past Sq.
__device__ __forceinline__ int kv_tiles_of(int qt, const FwdGeom& g, int causal) {
  if (qt * kTile >= g.Sq) return 0;
  if (!causal) return g.n_ktiles;
  const int last_row = min(g.Sq - 1, qt * kTile + kTile - 1);
  return (g.koff + last_row) / kTile + 1;
}

// The number of parts of a pair whose tile A visits nA key tiles (split forward).
__device__ __forceinline__ int fwd_pair_parts(int nA, int kcap) { return nA > kcap ? (nA + kcap - 1) / kcap : 1; }

__device__ __forceinline__ FwdSplitPos fwd_split_pos(int y, const FwdGeom& g, int causal, int n_pairs, int kcap) {
  int pidx = 0;
  for (int pr = n_pairs - 1; pr >= 0; --pr) {  // longest pairs first
    const int parts = fwd_pair_parts(kv_tiles_of(2 * pr, g, causal), kcap);
    if (y < parts) return FwdSplitPos{pr, y, parts, pidx};
    y -= parts;
    if (parts > 1) pidx += parts;
  }
  return FwdSplitPos{0, 0, 0, 0};  // past the plan (no such grid row is launched)
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
  griddep_wait();
  griddep_launch_dependents();

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int bh = blockIdx.x;                                   // b * Hq + h
  FwdGeom g;
  if (!fwd_geom(p, bh, g)) {
    if (tid == 0) atomicOr(p.status, STATUS_BAD_SEQLENS);
    return;
  }
  // Query-tile pair (longest pairs first) and, in a split forward, the part of its key range.
  FwdSplitPos sp{(int)gridDim.y - 1 - (int)blockIdx.y, 0, 1, 0};
  if (p.kcap > 0) sp = fwd_split_pos((int)blockIdx.y, g, p.causal, p.n_pairs, p.kcap);
  if (sp.parts == 0) return;
  const int pair = sp.pair;
  const int qtA = 2 * pair, qtB = 2 * pair + 1;
  const int nA_all = kv_tiles_of(qtA, g, p.causal);
  const int nB_all = kv_tiles_of(qtB, g, p.causal);
  if (nA_all == 0) return;  // a packed batch's short sequence: no query tile of this CTA exists
  // This CTA's key tiles kb .. kb + n_kv - 1 (all of them unless the pair is split: part q takes
  // [q nA / parts, (q + 1) nA / parts), the last part up to tile B's last key tile). Below, key
  // tiles are numbered from kb: nA, nB count tile A's and tile B's tiles in the range.
  const int n_all = nA_all > nB_all ? nA_all : nB_all;
  const int kb = sp.parts == 1 ? 0 : (int)((long long)sp.part * nA_all / sp.parts);
  const int ke = sp.part == sp.parts - 1 ? n_all : (int)((long long)(sp.part + 1) * nA_all / sp.parts);
  const int nA = (nA_all < ke ? nA_all : ke) - kb;  // >= 1: every part holds a key tile of tile A
  const int nB = nB_all > 0 ? (nB_all < ke ? nB_all : ke) - kb : 0;
  const int n_kv = ke - kb;
  const WaitGuard wg{&bars->abort_flag, p.status, kWaitLimitNs};
  // Extents of the tensors this CTA addresses, for the debug build's coordinate checks: heads of
  // the query / key maps and their rows (a packed CTA stays within its own sequence's rows).
  const int heads_q = p.cu_q ? p.Hq : (int)gridDim.x;
  const int heads_kv = p.cu_q ? p.Hkv : (int)gridDim.x / (p.Hq / p.Hkv);
  const int rows_q = p.cu_q ? p.Tq : p.Sq;

  if (tid == 0) {
    mbar_init(&bars->q_full[0], 1);
    mbar_init(&bars->q_full[1], 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < VST; ++s) mbar_init(&bars->v_empty[s], 1);
    mbar_init(&bars->k0_full, 1);
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
    // Q_A and K_0, which the first S product waits for, go out before the rest of the setup
    // (TMEM allocation, the block barrier, the register split); the producer takes over from Q_B.
    mbar_arrive_expect_tx(&bars->q_full[0], C::kTileBytes);
    mbar_arrive_expect_tx(&bars->k0_full, C::kTileBytes);
    const int qr = g.q_row0 + qtA * kTile, kr = g.k_row0 + kb * kTile;
    for (int c = 0; c < C::kChunks; ++c) {
      tma_load_3d_chk(smem + C::kQOff + c * kBoxBytes, &map_q, &bars->q_full[0], c * kChunk, qr, g.q_coord,
                      dbg_tile(c * kChunk, qr, g.q_coord, D, kChunk, g.q_row0, g.q_row0 + g.Sq, heads_q, p.status));
      tma_load_3d_chk(smem + C::kKOff + c * kBoxBytes, &map_k, &bars->k0_full, c * kChunk, kr, g.kv_coord,
                      dbg_tile(c * kChunk, kr, g.kv_coord, D, kChunk, g.k_row0, g.k_row0 + g.Sk, heads_kv, p.status));
    }
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
    // ------------------------------------------------------------ TMA producer: Q, then the K and V rings
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      // Q_A and K_0 came from thread 0; then Q_B (only when tile B has rows; its buffer is
      // otherwise never read), then V_0: the first S products wait for Q and K_0 only.
      auto load_q = [&](int t) {
        mbar_arrive_expect_tx(&bars->q_full[t], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          const int r = g.q_row0 + (qtA + t) * kTile;
          tma_load_3d_chk(smem + C::kQOff + t * C::kTileBytes + c * kBoxBytes, &map_q, &bars->q_full[t], c * kChunk,
                          r, g.q_coord,
                          dbg_tile(c * kChunk, r, g.q_coord, D, kChunk, g.q_row0, g.q_row0 + g.Sq, heads_q, p.status));
        }
      };
      bool q_b_issued = false;
      int issued = 0;
      // K_j and V_j land on one barrier, kv_full[j % ST]: the MMA issuer waits once per key tile.
      // A stage of K is reused only after both S products that read it completed, which comes
      // after the issuer's wait on that barrier's previous phase.
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % ST, vst = j % VST;
        if (j >= ST && !mbar_wait(&bars->k_empty[st], ((j / ST) - 1) & 1, wg)) break;
        if (j >= VST && !mbar_wait(&bars->v_empty[vst], ((j / VST) - 1) & 1, wg)) break;
        mbar_arrive_expect_tx(&bars->kv_full[st], (j == 0 ? 1 : 2) * C::kTileBytes);
        const int r = g.k_row0 + (kb + j) * kTile;
        if (j > 0)  // K_0 is on its way already
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d_chk(smem + C::kKOff + st * C::kTileBytes + c * kBoxBytes, &map_k, &bars->kv_full[st],
                            c * kChunk, r, g.kv_coord,
                            dbg_tile(c * kChunk, r, g.kv_coord, D, kChunk, g.k_row0, g.k_row0 + g.Sk, heads_kv,
                                     p.status));
        if (j == 0 && nB > 0) {  // Q_B between K_0 and V_0
          load_q(1);
          q_b_issued = true;
        }
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d_chk(smem + C::kVOff + vst * C::kTileBytes + c * kBoxBytes, &map_v, &bars->kv_full[st],
                          c * kChunk, r, g.kv_coord,
                          dbg_tile(c * kChunk, r, g.kv_coord, D, kChunk, g.k_row0, g.k_row0 + g.Sk, heads_kv,
                                   p.status));
        issued = j + 1;
        if (j == 0 && p.n_sm > 0 && p.kcap == 0 && p.cu_q == nullptr) {
          // The query tiles of the CTA one wave later (grid position + n_sm, where it will most
          // likely start as this wave's CTAs finish) into L2: its own first loads then come from
          // L2 rather than DRAM.
          const int nxt = (int)(blockIdx.y * gridDim.x + blockIdx.x) + p.n_sm;
          if (nxt < (int)(gridDim.x * gridDim.y)) {
            const int y2 = nxt / (int)gridDim.x;
            const int bh2 = nxt - y2 * (int)gridDim.x;
            const int row2 = (2 * ((int)gridDim.y - 1 - y2)) * kTile;
            for (int t = 0; t < 2; ++t)
              if (row2 + t * kTile < p.Sq)
                for (int c = 0; c < C::kChunks; ++c) tma_prefetch_l2_3d(&map_q, c * kChunk, row2 + t * kTile, bh2);
          }
        }
      }
      if (bars->abort_flag) {
        // Let every copy already issued land before the CTA's shared memory goes away.
        mbar_wait_drain(&bars->q_full[0], 0, kWaitLimitNs);
        if (q_b_issued) mbar_wait_drain(&bars->q_full[1], 0, kWaitLimitNs);
        mbar_wait_drain(&bars->k0_full, 0, kWaitLimitNs);  // K_0 was issued with Q_A
        for (int j = (issued > ST ? issued - ST : 0); j < issued; ++j)
          mbar_wait_drain(&bars->kv_full[j % ST], (j / ST) & 1, kWaitLimitNs);
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
      // O_X += P_X(j) V_j, P_X(j) read from the S columns of tile X. O_X is signalled complete
      // after its last product only: within the loop, S_X(j + 1) completing (issued after
      // P_X(j) V_j by this thread) already tells the softmax warps that O_X holds P_X(j) V_j.
      auto issue_pv = [=](int x, int j, bool last) {
        const uint64_t bv = dv0 + (uint64_t)(j % VST) * kTileDesc;
        const uint32_t p_tmem = tbase + (uint32_t)x * 128u;
        const uint32_t o_tmem = tbase + C::kOCol + (uint32_t)x * D;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts(o_tmem, p_tmem + (uint32_t)kk * 8u, bv + (uint64_t)((kk * 2048) >> 4), idesc_o,
                  (j > 0 || kk > 0) ? 1u : 0u);
        if (last) umma_commit(&bars->o_done[x]);
      };
      // K_j is released once the last S MMA reading it completes, V_j once both P V MMAs do:
      // the K ring refills a full key tile earlier than a shared K/V stage would. Each key tile
      // costs one wait (kv_full) here: a wait on a barrier, even one already complete, stalls
      // this thread for a few hundred cycles, and the tensor core holds about one MMA in its queue.
      bool ok = mbar_wait(&bars->q_full[0], 0, wg) && mbar_wait(&bars->k0_full, 0, wg);
      if (kRope && ok) ok = mbar_wait(&bars->q_ready[0], 0, wg);  // the softmax warps rotate their queries first
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);  // nA > 0 for every CTA that gets here
      }
      if (ok && nB > 0) {
        ok = mbar_wait(&bars->q_full[1], 0, wg) && (!kRope || mbar_wait(&bars->q_ready[1], 0, wg));
        if (ok) {
          tc_fence_after();
          issue_s(1, 0);
        }
      }
      // V_j landed with K_j, before S(j) was issued: P(j) V_j needs no wait of its own, but V_0
      // does. Its wait comes before K_0's stage is released: the producer arms kv_full[0] again
      // for K_ST only after that release, and arming a barrier whose phase is still open would
      // add an arrival that phase does not expect.
      if (ok) ok = mbar_wait(&bars->kv_full[0], 0, wg);
      if (ok) umma_commit(&bars->k_empty[0]);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int vst = j % VST;
        const int j1 = j + 1;
        const int st1 = j1 % ST;
        if (j < nA) {
          if (!(ok = mbar_wait(&bars->p_full[0], j & 1, wg))) break;
          tc_fence_after();
          issue_pv(0, j, j1 == nA);
          if (j1 < nA) {
            if (!(ok = mbar_wait(&bars->kv_full[st1], (j1 / ST) & 1, wg))) break;
            tc_fence_after();
            issue_s(0, j1);
          }
        }
        if (j < nB) {
          if (!(ok = mbar_wait(&bars->p_full[1], j & 1, wg))) break;
          tc_fence_after();
          issue_pv(1, j, j1 == nB);
          if (j1 < nB) {  // K_{j+1} and V_{j+1} were already waited for when tile A uses them too
            if (j1 >= nA && !(ok = mbar_wait(&bars->kv_full[st1], (j1 / ST) & 1, wg))) break;
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
    // Running reference max and sum; the reference is taken from the first key tile in which the
    // row sees a key (a part of a split key range can start with a tile the row does not see yet).
    float m_ref = 0.f, l = 0.f;
    bool have_ref = false;
    bool ok = true;
    if (kRope && n_x > 0) {
      // Rotary embedding: each thread turns its own query row of tile X in shared memory
      // (rows past S hold zeros and have no table row).
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full[x], 0, wg));
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

      const int kv0 = (kb + j) * kTile;  // the key tile's first key
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
      if (!have_ref) {
        if (m_tile > -INFINITY) {
          m_ref = m_tile;
          have_ref = true;
        }
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
        // O_X holds the sum up to tile j-1 against the old reference: P_X(j-1) V_{j-1} completed
        // before S_X(j) did (one thread issued both, in that order, and the commit that signalled
        // S_X(j) tracks every MMA it issued before).
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
    if (ok && n_x > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done[x], 0, wg));
    if (ok && n_x > 0 && sp.parts > 1) {
      // Split key range: this part's unnormalised O tile X and its (m, l) go to the part's slot
      // (m = -inf for a row that saw no key in the range). A warp's stores cover 32 consecutive
      // rows of one float4 column: 512 contiguous bytes.
      tc_fence_after();
      const size_t slot_fl = fwd_slot_floats(D);
      float* tile = p.part + ((size_t)bh * p.parts_per_bh + sp.pidx + sp.part) * slot_fl +
                    (size_t)x * (slot_fl / 2);
      const long long slot_end = (long long)gridDim.x * p.parts_per_bh * (long long)slot_fl;
      if (dbg_range((long long)(tile - p.part), (long long)(slot_fl / 2), slot_end, p.status) &&
          dbg_ok((reinterpret_cast<uintptr_t>(tile) & 15u) == 0, p.status)) {
        float4* cols = reinterpret_cast<float4*>(tile);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(o_tmem + cc * 32, o);
          tmem_wait_ld_x32(o);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            cols[(size_t)(cc * 8 + u) * kTile + row] =
                make_float4(__uint_as_float(o[4 * u]), __uint_as_float(o[4 * u + 1]), __uint_as_float(o[4 * u + 2]),
                            __uint_as_float(o[4 * u + 3]));
        }
        tile[(size_t)kTile * D + row] = have_ref ? m_ref : -INFINITY;
        tile[(size_t)kTile * D + kTile + row] = l;
      }
    } else if (ok && n_x > 0) {
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

// Key tiles query tile qt of a dense batch sees (kv_tiles_of without the per-CTA geometry).
__host__ __device__ inline int dense_kv_tiles(int qt, int Sq, int Sk, int causal) {
  if (qt * kTile >= Sq) return 0;
  const int n_ktiles = (Sk + kTile - 1) / kTile;
  if (!causal) return n_ktiles;
  const int last_row = Sq - 1 < qt * kTile + kTile - 1 ? Sq - 1 : qt * kTile + kTile - 1;
  return (Sk - Sq + last_row) / kTile + 1;
}

struct FwdCombineParams {
  const float* part;
  uint16_t* o;  // [B*Hq, Sq, D] bf16
  float* lse;   // [B*Hq, Sq]
  int Sq, Sk, causal, kcap, n_pairs, parts_per_bh;
  int* status;
};

// Merge of a split forward's parts: for row r of a tile cut into parts p with maxima m_p, sums
// l_p and unnormalised rows O_p, M = max m_p, L = sum l_p 2^(m_p - M), O = sum O_p 2^(m_p - M) / L,
// LSE = (M + log2 L) ln 2; parts are added in part order, so the result is reproducible. One CTA
// takes 128 rows x 8 columns of one tile of one split pair: grid x = batch entry x head, grid y =
// (split pair, tile, column chunk). A warp's loads cover 32 rows of one float4 column of a slot
// (512 contiguous bytes); the part loops are unrolled so that a thread has many loads in flight.
template <int D>
__global__ void __launch_bounds__(128) fwd_combine_kernel(const FwdCombineParams p) {
  griddep_wait();  // the parts' slots are written by the forward just ahead
  griddep_launch_dependents();
  constexpr int kChunks = D / 8;
  const int bh = blockIdx.x;
  const int cchunk = (int)blockIdx.y % kChunks;
  const int x = ((int)blockIdx.y / kChunks) & 1;
  int s = (int)blockIdx.y / (2 * kChunks);
  const int row = threadIdx.x;
  // the s-th split pair, longest pairs first, and the index of its first slot
  int pair = -1, parts = 0, pidx = 0;
  for (int pr = p.n_pairs - 1; pr >= 0; --pr) {
    const int nA = dense_kv_tiles(2 * pr, p.Sq, p.Sk, p.causal);
    const int np = nA > p.kcap ? (nA + p.kcap - 1) / p.kcap : 1;
    if (np < 2) continue;
    if (s == 0) {
      pair = pr;
      parts = np;
      break;
    }
    --s;
    pidx += np;
  }
  if (pair < 0) return;
  const int qrow = (2 * pair + x) * kTile + row;
  if (qrow >= p.Sq) return;
  const size_t slot_fl = fwd_slot_floats(D);
  const float* tile = p.part + ((size_t)bh * p.parts_per_bh + pidx) * slot_fl + (size_t)x * (slot_fl / 2);
  const long long slot_end = (long long)gridDim.x * p.parts_per_bh * (long long)slot_fl;
  if (!dbg_range((long long)(tile - p.part) + (long long)(parts - 1) * (long long)slot_fl, (long long)(slot_fl / 2),
                 slot_end, p.status))
    return;
  const float* m_of = tile + (size_t)kTile * D + row;
  const float* l_of = m_of + kTile;
  // Loads are issued a group of parts at a time (predicated past the last part), then consumed.
  constexpr int kGroup = 4;
  float M = -INFINITY;
  for (int p0 = 0; p0 < parts; p0 += 2 * kGroup) {
    float mm[2 * kGroup];
#pragma unroll
    for (int i = 0; i < 2 * kGroup; ++i) mm[i] = p0 + i < parts ? m_of[(size_t)(p0 + i) * slot_fl] : -INFINITY;
#pragma unroll
    for (int i = 0; i < 2 * kGroup; ++i) M = fmaxf(M, mm[i]);
  }
  float L = 0.f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const float4* cols = reinterpret_cast<const float4*>(tile) + (size_t)cchunk * 2 * kTile + row;
  for (int p0 = 0; p0 < parts; p0 += kGroup) {  // part order
    float mm[kGroup], ll[kGroup];
    float4 a[kGroup], b[kGroup];
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      const size_t off = (size_t)(p0 + i) * slot_fl;
      const bool in = p0 + i < parts;
      mm[i] = in ? m_of[off] : -INFINITY;
      ll[i] = in ? l_of[off] : 0.f;
      a[i] = in ? cols[off / 4] : make_float4(0.f, 0.f, 0.f, 0.f);
      b[i] = in ? cols[off / 4 + kTile] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      const float w = ex2_approx(mm[i] - M);  // 0 for a part where the row saw no key, or none
      L = fmaf(ll[i], w, L);
      acc[0] = fmaf(a[i].x, w, acc[0]);
      acc[1] = fmaf(a[i].y, w, acc[1]);
      acc[2] = fmaf(a[i].z, w, acc[2]);
      acc[3] = fmaf(a[i].w, w, acc[3]);
      acc[4] = fmaf(b[i].x, w, acc[4]);
      acc[5] = fmaf(b[i].y, w, acc[5]);
      acc[6] = fmaf(b[i].z, w, acc[6]);
      acc[7] = fmaf(b[i].w, w, acc[7]);
    }
  }
  const float inv_l = 1.f / L;
  const long long orow_off = ((long long)bh * p.Sq + qrow) * D + cchunk * 8;
  if (dbg_range(orow_off, 8, (long long)gridDim.x * p.Sq * D, p.status))
    *reinterpret_cast<uint4*>(p.o + orow_off) =
        make_uint4(pack_bf16(acc[0] * inv_l, acc[1] * inv_l), pack_bf16(acc[2] * inv_l, acc[3] * inv_l),
                   pack_bf16(acc[4] * inv_l, acc[5] * inv_l), pack_bf16(acc[6] * inv_l, acc[7] * inv_l));
  if (cchunk == 0) p.lse[(size_t)bh * p.Sq + qrow] = (M + __log2f(L)) * 0.69314718055994530942f;
}

// Plan of the split forward. A CTA's time is modelled in key-tile units (one 128 x 128 tile of one
// query tile, about 0.9 us at D = 128): its units, plus kFwdCtaOverheadUnits (prologue, epilogue),
// plus kFwdPartWriteUnits for a part of a split pair (its slot write). CTAs are dealt longest first
// onto kPlanCtas SMs; a split grid adds the combine kernel, kFwdCombineLaunchUnits plus one unit per
// kFwdCombineBytesPerUnit of slots it reads. The kcap with the shortest estimate wins if it beats
// the unsplit grid by kFwdSplitGain; only problems whose unsplit grid has at most two waves split.
constexpr int kFwdCtaOverheadUnits = 4;
constexpr int kFwdPartWriteUnits = 2;
constexpr int kFwdCombineLaunchUnits = 4;
constexpr long long kFwdCombineBytesPerUnit = 3ll << 20;
constexpr double kFwdSplitGain = 1.15;

long long fwd_plan_makespan(int BH, int Sq, int Sk, int causal, int D, int n_pairs, int kcap) {
  std::vector<int> sizes;
  long long slots = 0;  // per (batch entry, head)
  for (int pr = 0; pr < n_pairs; ++pr) {
    const int nA = dense_kv_tiles(2 * pr, Sq, Sk, causal), nB = dense_kv_tiles(2 * pr + 1, Sq, Sk, causal);
    if (nA == 0) continue;
    const int n_all = nA > nB ? nA : nB;
    const int parts = kcap > 0 && nA > kcap ? ceil_div(nA, kcap) : 1;
    if (parts > 1) slots += parts;
    for (int q = 0; q < parts; ++q) {
      const int kb = (int)((long long)q * nA / parts);
      const int ke = q == parts - 1 ? n_all : (int)((long long)(q + 1) * nA / parts);
      int units = kFwdCtaOverheadUnits + (parts > 1 ? kFwdPartWriteUnits : 0);
      for (int j = kb; j < ke; ++j) units += (j < nA) + (j < nB);
      for (int h = 0; h < BH; ++h) sizes.push_back(units);
    }
  }
  std::sort(sizes.begin(), sizes.end(), std::greater<int>());
  std::priority_queue<long long, std::vector<long long>, std::greater<long long>> load;
  for (int i = 0; i < kPlanCtas; ++i) load.push(0);
  long long span = 0;
  for (int sz : sizes) {
    const long long t = load.top() + sz;
    load.pop();
    load.push(t);
    span = t > span ? t : span;
  }
  if (slots > 0)
    span += kFwdCombineLaunchUnits +
            (long long)(slots * BH * fwd_slot_floats(D) * sizeof(float)) / kFwdCombineBytesPerUnit;
  return span;
}

FwdSplit fwd_split_plan_uncached(int BH, int Sq, int Sk, int causal, int D) {
  const int n_pairs = ceil_div(Sq, 2 * kTile);
  FwdSplit sp{0, n_pairs, n_pairs, 0, 0};
  const int nA_first = dense_kv_tiles(0, Sq, Sk, causal), nA_last = dense_kv_tiles(2 * (n_pairs - 1), Sq, Sk, causal);
  const int nA_max = nA_last > nA_first ? nA_last : nA_first;
  if ((long long)BH * n_pairs > 2ll * kPlanCtas || nA_max < 2) return sp;
  const long long unsplit = fwd_plan_makespan(BH, Sq, Sk, causal, D, n_pairs, 0);
  long long best = unsplit;
  int best_cap = 0;
  for (int cap = nA_max - 1; cap >= 1; --cap) {
    // Grids of more than four waves are not considered; smaller caps only add CTAs, so the
    // search (and its host time on a first call) stops there.
    long long ctas = 0;
    for (int pr = 0; pr < n_pairs; ++pr) {
      const int nA = dense_kv_tiles(2 * pr, Sq, Sk, causal);
      ctas += nA > cap ? ceil_div(nA, cap) : (nA > 0 ? 1 : 0);
    }
    if ((long long)BH * ctas > 4ll * kPlanCtas) break;
    const long long m = fwd_plan_makespan(BH, Sq, Sk, causal, D, n_pairs, cap);
    if (m < best) {
      best = m;
      best_cap = cap;
    }
  }
  if (best_cap == 0 || (double)best * kFwdSplitGain > (double)unsplit) return sp;
  sp.kcap = best_cap;
  sp.ctas_y = 0;
  for (int pr = 0; pr < n_pairs; ++pr) {
    const int nA = dense_kv_tiles(2 * pr, Sq, Sk, causal);
    const int parts = nA > best_cap ? ceil_div(nA, best_cap) : 1;
    sp.ctas_y += parts;
    if (parts > 1) {
      sp.parts_per_bh += parts;
      ++sp.split_pairs;
    }
  }
  return sp;
}

}  // namespace

FwdSplit fwd_split_plan(int BH, int Sq, int Sk, int causal, int D) {
  struct Entry {
    int key[5];
    FwdSplit plan;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  const int key[5] = {BH, Sq, Sk, causal ? 1 : 0, D};
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry& e : cache)
      if (std::equal(key, key + 5, e.key)) return e.plan;
  }
  const FwdSplit plan = fwd_split_plan_uncached(BH, Sq, Sk, causal, D);
  std::lock_guard<std::mutex> lk(mu);
  if (cache.size() < 256) cache.push_back(Entry{{key[0], key[1], key[2], key[3], key[4]}, plan});
  return plan;
}

FwdWorkspace fwd_workspace_layout(int B, int Hq, int Sq, int Sk, int D) {
  FwdWorkspace w{0};
  int slots = 0;
  for (int causal = 0; causal < 2; ++causal) {
    const FwdSplit sp = fwd_split_plan(B * Hq, Sq, Sk, causal, D);
    if (sp.kcap > 0 && sp.parts_per_bh > slots) slots = sp.parts_per_bh;
  }
  if (slots > 0) w.total = align256((size_t)B * Hq * slots * fwd_slot_floats(D) * sizeof(float));
  return w;
}

namespace {

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
  p.G = a.Hq / a.Hkv;
  p.div_hq = udiv_magic(a.Hq);
  p.div_g = udiv_magic(p.G);
  const size_t q_bytes = (size_t)a.B * a.Hq * a.Sq * a.D * 2;
  p.n_sm = 2 * q_bytes <= (size_t)device_l2_bytes() ? device_sm_count() : 0;
  p.status = a.status;
  // Dense forward given a split workspace: the key ranges of the longest pairs may be split.
  const FwdSplit split = (a.part && !a.cu_q) ? fwd_split_plan(a.B * a.Hq, a.Sq, a.Sk, a.causal, D)
                                             : FwdSplit{0, ceil_div(a.Sq, 2 * kTile), ceil_div(a.Sq, 2 * kTile), 0, 0};
  p.kcap = split.kcap;
  p.n_pairs = split.n_pairs;
  p.parts_per_bh = split.parts_per_bh;
  p.part = a.part;
  auto kern = a.rope_cos ? fwd_kernel<D, true> : fwd_kernel<D, false>;
  // The setmaxnreg split must fit the registers the block is launched with, or the
  // increase would wait forever: kernel_setup refuses the launch otherwise.
  cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads,
                               2 * 128 * C::kHighRegs + 128 * C::kLowRegs);
  if (e != cudaSuccess) return e;
  // Packed batch: one row of CTAs per (sequence, head), enough pairs for the longest sequence.
  const int rows = a.cu_q ? a.max_seqlen_q : a.Sq;
  dim3 grid((unsigned)(a.B * a.Hq), (unsigned)(split.kcap > 0 ? split.ctas_y : ceil_div(rows, 2 * kTile)));
  trace_begin(kKernelFwd, stream);
  e = launch_pdl(kern, grid, dim3(C::kThreads), C::kSmemBytes, stream, *a.map_q, *a.map_k, *a.map_v, *a.map_o, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  trace_end(kKernelFwd, stream);
  if (e != cudaSuccess || split.split_pairs == 0) return e;
  // The split pairs' slots are merged into O and LSE.
  FwdCombineParams cp;
  cp.part = a.part;
  cp.o = static_cast<uint16_t*>(a.o);
  cp.lse = a.lse;
  cp.Sq = a.Sq;
  cp.Sk = a.Sk;
  cp.causal = a.causal;
  cp.kcap = split.kcap;
  cp.n_pairs = split.n_pairs;
  cp.parts_per_bh = split.parts_per_bh;
  cp.status = a.status;
  const dim3 cgrid((unsigned)(a.B * a.Hq), (unsigned)(split.split_pairs * 2 * (D / 8)));
  trace_begin(kKernelFwdCombine, stream);
  e = launch_pdl(fwd_combine_kernel<D>, cgrid, dim3(128), 0, stream, cp);
  if (e == cudaSuccess) e = cudaGetLastError();
  trace_end(kKernelFwdCombine, stream);
  return e;
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.D == 64) return launch_fwd_d<64>(a, stream);
  return launch_fwd_d<128>(a, stream);
}

}  // namespace gqa
