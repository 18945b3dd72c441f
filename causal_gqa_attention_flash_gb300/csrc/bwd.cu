// Backward of fused causal grouped-query attention on sm_103a.
//
// The gradient of a comprehension is itself a comprehension, so the backward
// writes no S x S intermediate either (aiinsiders.net, "A compiler that
// derives GPU kernels matches hand-tuned code"); every contraction
// accumulates in f32 (the same article reports a bf16-accumulating fused
// backward failing the f32 tolerance). Three kernels on one stream:
//
//   bwd_prep      D_i = sum_d dO_id O_id (f32), -LSE_i * log2(e) (-inf past S),
//                 and a zeroed f32 dQ accumulator;                    HBM-bound
//   bwd_main      one CTA per (batch, KV head, 128-key tile). For every query
//                 head of the group and every query tile that can see the key
//                 tile it recomputes S^T = K Q^T, P^T = exp2(S^T c - LSE2),
//                 dP^T = V dO^T, dS^T = P^T (dP^T - D), and accumulates
//                 dV += P^T dO and dK += dS^T Q in TMEM (so the GQA reduction
//                 over the group happens inside the CTA, in a fixed order:
//                 dK/dV are deterministic), and dQ_i += dS K by a TMA
//                 reduce-add of the f32 partial into the accumulator;
//   bwd_convert   dQ = bf16(scale * accumulator);                     HBM-bound
//
// bwd_main warp roles are listed above the kernel; element-wise thread r of a
// lane quarter owns TMEM lane r (key row r for S^T, dP^T, dK, dV; query row r
// for the dQ partial).
// TMEM columns: [0,128) S^T f32; column half h (query columns [64h, 64h+64))
// then holds its packed bf16 P^T in [64h, 64h+32) and dS^T in [64h+32, 64h+64),
// written only by the warpgroup that read those S^T columns; [128,256) dP^T
// f32, then the dQ partial f32 [128, 128+D); [256,256+D) dV; [256+D,256+2D) dK.
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

__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ------------------------------------------------------------------ prep

// One group of D/8 threads per row: each thread reads 8 bf16 of dO and of O. Rows of the padded
// arrays past rows_valid, or with s >= S, are padding (D = 0, -LSE2 = -inf).
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dO,
                                                       const float* __restrict__ lse, float* __restrict__ dvec,
                                                       float* __restrict__ nlse2, float* __restrict__ dq_acc,
                                                       int rows_total, int rows_valid, int S, int S_pad,
                                                       float log2e, long long acc_vec4, unsigned* tickets,
                                                       int n_tickets, int* status) {
  constexpr int TPR = D / 8;            // threads per row
  constexpr int RPW = 32 / TPR;          // rows per warp and iteration
  griddep_wait();  // O and LSE come from the forward, which may be just ahead in the stream
  griddep_launch_dependents();
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nthreads = gridDim.x * blockDim.x;
  const int lane = threadIdx.x & 31;
  const int sub = lane % TPR;
  // Rows of the padded [B*Hq, S_pad] arrays; the loop bound is warp-uniform so
  // that every lane takes part in the shuffles.
  for (int r0 = (gtid >> 5) * RPW; r0 < rows_total; r0 += (nthreads >> 5) * RPW) {
    const int r = r0 + lane / TPR;
    const int bh = r / S_pad;
    const int s = r - bh * S_pad;
    const bool live = r < rows_total;
    const bool real = r < rows_valid && s < S;  // a row of O / dO (not padding)
    float acc = 0.f;
    if (live && real && dbg_range(((long long)bh * S + s) * D + sub * 8, 8, (long long)(rows_valid / S_pad) * S * D,
                                  status)) {
      const size_t base = ((size_t)bh * S + s) * D + sub * 8;
      const uint4 a = *reinterpret_cast<const uint4*>(o + base);
      const uint4 b = *reinterpret_cast<const uint4*>(dO + base);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc = fmaf(__uint_as_float(aw[i] << 16), __uint_as_float(bw[i] << 16), acc);
        acc = fmaf(__uint_as_float(aw[i] & 0xFFFF0000u), __uint_as_float(bw[i] & 0xFFFF0000u), acc);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, TPR);
    if (live && sub == 0 && dbg_range(r, 1, rows_total, status)) {
      dvec[r] = acc;
      nlse2[r] = real ? -(lse[(size_t)bh * S + s] * log2e) : -INFINITY;
    }
  }
  float4* acc4 = reinterpret_cast<float4*>(dq_acc);
  for (long long i = gtid; i < acc_vec4; i += nthreads) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = gtid; i < n_tickets; i += nthreads) tickets[i] = 0u;  // split key tiles' arrival counters
}

// ------------------------------------------------------------------ convert

__global__ void __launch_bounds__(256) bwd_convert_kernel(const float* __restrict__ dq_acc, uint16_t* __restrict__ dq,
                                                          long long n8, float scale) {
  griddep_wait();  // the accumulator is complete once the main kernel ahead of this one is
  griddep_launch_dependents();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * i + 1];
    uint4 w;
    w.x = pack_bf16(a.x * scale, a.y * scale);
    w.y = pack_bf16(a.z * scale, a.w * scale);
    w.z = pack_bf16(b.x * scale, b.y * scale);
    w.w = pack_bf16(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = w;
  }
}

// ------------------------------------------------------------------ main

template <int D>
struct BwdCfg {
  static constexpr int kChunks = D / kChunk;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = 2;                                    // Q / dO ring
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;
  static constexpr int kDOOff = kQOff + kStages * kTileBytes;
  static constexpr int kDSOff = kDOOff + kStages * kTileBytes;         // dS bf16 [128 kv][128 q], MN-major
  static constexpr int kDSBytes = kTile * kTile * 2;
  static constexpr int kRowOff = kDSOff + kDSBytes;                    // per stage: -LSE2, D rows
  static constexpr int kRowFl = 136;                                   // floats per row buffer (>= 4 + 128)
  static constexpr int kBarOff = kRowOff + kStages * 2 * kRowFl * 4;
  static constexpr int kSmemBytes = kBarOff + 256;                     // the base is checked to be 1024-aligned
  static constexpr int kThreads = 352;
  static constexpr int kRounds = D / 64;                               // 32-column dQ slices per warpgroup
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSPCol = 0, kDPCol = 128, kDVCol = 256, kDKCol = 256 + D;
};

template <int ST>
struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[ST];   // Q(t) and the step's -LSE2 / D rows landed
  uint64_t do_full[ST];  // dO(t) landed
  uint64_t q_empty[ST];  // the Q stage may be refilled
  uint64_t do_empty[ST]; // the dO stage may be refilled
  uint64_t s_full, dp_full, p_full, ds_full, dq_full, dq_free, stage_full, dkv_done, drain;
  uint64_t k_ready;  // rotary embedding: the key tile rotated in shared memory
  uint64_t epi_bar;  // split key tiles: barrier of the element-wise warps around the partials' ticket
  uint32_t tmem_base;
  int abort_flag;
  int last;          // split key tiles: this part arrived last and adds the parts up
};

static_assert(sizeof(BwdBars<BwdCfg<64>::kStages>) <= 256 && sizeof(BwdBars<BwdCfg<128>::kStages>) <= 256,
              "backward barriers exceed the 256 bytes reserved for them");
static_assert(BwdCfg<64>::kSmemBytes <= 232448 && BwdCfg<128>::kSmemBytes <= 232448, "backward smem over the limit");

struct BwdKParams {
  const float* nlse2;  // -LSE * log2(e) rows
  const float* dvec;
  uint16_t* dk;
  uint16_t* dv;
  const int* cu;  // packed batch: sequence bounds (nullptr: dense batch)
  // Dense: S rows per (b, head), D / LSE2 rows padded to S_pad per head. Packed: S = total rows
  // T, row stride of D / LSE2 = T (S_pad = T), sequences of at most max_seqlen rows.
  int Hq, Hkv, S, S_pad, causal, max_seqlen;
  int n_ktiles;   // packed batch: key tiles of the longest sequence (the 1-D grid's inner extent)
  int rows_total; // rows of the D / LSE2 arrays (padding included)
  // Dense batches with split key tiles (cap > 0): grid y enumerates each group's (key tile, part)
  // pairs, ctas_per_group of them; a group keeps parts_per_group f32 dK / dV partials in `part`.
  int cap, ctas_per_group, parts_per_group;
  float* part;
  unsigned* tickets;
  float scale, scale_log2;
  int* status;
  const float* rope_cos;  // rotary tables [S, D/2] (nullptr: none): K is rotated in shared memory,
  const float* rope_sin;  // the queries arrive rotated, dK is turned back in the epilogue
};

// Position of grid row x among a group's (key tile, part) pairs when key tiles are split (see
// BwdSplit): key tile jt has ceil(steps(jt) / cap) parts; pidx is the index of the tile's first
// partial among the group's partials (only split key tiles keep partials).
struct SplitPos {
  int jt, part, parts, pidx;
};

__device__ __forceinline__ SplitPos split_pos(int x, int n_tiles, int G, int causal, int cap) {
  int pidx = 0;
  for (int jt = 0; jt < n_tiles; ++jt) {
    const int parts = (G * (causal ? n_tiles - jt : n_tiles) + cap - 1) / cap;
    if (x < parts) return SplitPos{jt, x, parts, pidx};
    x -= parts;
    if (parts > 1) pidx += parts;
  }
  return SplitPos{n_tiles, 0, 1, 0};  // past the plan (no such grid row is launched)
}

// One CTA per (batch, KV head, 128-key tile jt), 352 threads:
//   warps 0..7  element-wise work. Warp w owns TMEM lane quarter w % 4 (key
//               rows of S^T, dP^T, dK, dV; query rows of the dQ partial) and the
//               column half h = w / 4 (query columns [64h, 64h+64) of S^T / dP^T;
//               dQ / dK / dV columns of that half);
//   warp 8      TMA producer: K, V once; Q, dO, LSE2 and D rows per step, 2 stages;
//   warp 9      MMA issuer (one thread) and TMEM owner;
//   warp 10     dQ reduce: TMA reduce-add of each step's staged dQ partial.
// A step is one (query head of the group, query tile i). MMA order per step t:
//   dV(t) after P(t) is written, dK(t) and dQ(t) after dS(t) is written, then at
//   once S(t+1) (its Q is already staged) and, once the dQ(t) columns have been
//   read out, dP(t+1). The element-wise warps load the dQ partial into registers,
//   release its TMEM columns, and only then stage it, in one round, into this
//   step's Q and dO tiles (free once dQ(t) has completed). Warp 10 issues the TMA
//   reduce-adds, waits until they have read the staging and hands the Q/dO stage
//   back to the producer; the reduce streams out while the next step runs.
// kDq = false: the deterministic backward's dK/dV kernel. It skips the dQ partial (a
// query-major kernel computes dQ); the Q/dO stage is released once dK and dV have read it.
// kRope: the key tile is turned by the rotary embedding in shared memory (the queries arrive
// rotated) and dK is turned back in the epilogue. kPacked: a packed batch of variable-length
// sequences (bounds read per CTA, query columns past the sequence masked explicitly, D / LSE2
// rows copied from an aligned start).
template <int D, bool kDq, bool kRope, bool kPacked>
__global__ void __launch_bounds__(352, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                    const __grid_constant__ CUtensorMap map_acc, const BwdKParams p) {
  using C = BwdCfg<D>;
  constexpr int ST = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  auto* bars = reinterpret_cast<BwdBars<ST>*>(smem + C::kBarOff);
  griddep_wait();  // the D / -LSE2 rows and the zeroed accumulator come from the kernel ahead
  griddep_launch_dependents();

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // The 128-byte swizzled tiles need a 1024-byte aligned base; report instead of faulting.
  if ((smem_addr(smem) & 1023u) != 0) {
    if (tid == 0) atomicOr(p.status, STATUS_MISALIGNED_SMEM);
    return;
  }
  // Key tile jt (tile 0 sees the most query tiles when causal) of group grp = (batch entry or
  // sequence, KV head). Dense: grid (groups, key tiles), the groups fastest, so that each wave
  // holds ~9 neighbouring key tiles of every group. Packed: a 1-D grid that walks each group's key
  // tiles consecutively, so that a sequence's key tiles run together and share its Q, dO and
  // dQ-accumulator tiles in L2; with the groups fastest, a wave would hold about one key tile of
  // every sequence and nearly every load and reduce-add would go to DRAM.
  // Dense batches with split key tiles: grid y is the (key tile, part) pair of the group.
  const int G = p.Hq / p.Hkv;
  SplitPos sp{kPacked ? (int)(blockIdx.x % (unsigned)p.n_ktiles) : (int)blockIdx.y, 0, 1, 0};
  if (!kPacked && p.cap > 0) sp = split_pos((int)blockIdx.y, p.n_ktiles, G, p.causal, p.cap);
  const int jt = sp.jt;
  const int grp = kPacked ? (int)(blockIdx.x / (unsigned)p.n_ktiles) : (int)blockIdx.x;
  const int b = grp / p.Hkv;  // batch entry (dense) or sequence (packed)
  const int hkv = grp - b * p.Hkv;
  // L rows in this CTA's sequence, starting at row0 of the tensor maps; the KV head's map
  // coordinate, the first query head's, and the row stride of the D / LSE2 arrays.
  int L, row0, kv_coord, bhq0;
  if (!kPacked) {
    L = p.S;
    row0 = 0;
    kv_coord = grp;
    bhq0 = b * p.Hq + hkv * G;
  } else {
    const int s0 = __ldg(p.cu + b), s1 = __ldg(p.cu + b + 1);
    if (s0 < 0 || s1 < s0 || s1 > p.S || s1 - s0 > p.max_seqlen) {
      if (tid == 0) atomicOr(p.status, STATUS_BAD_SEQLENS);
      return;
    }
    L = s1 - s0;
    row0 = s0;
    kv_coord = hkv;
    bhq0 = hkv * G;
  }
  if (jt * kTile >= L) return;  // a packed batch's short sequence: this key tile does not exist
  // Extents for the debug build's coordinate checks: heads of the query and key maps, and the
  // rows of this CTA's sequence.
  const int heads_q = kPacked ? p.Hq : (int)gridDim.x * G;
  const int heads_kv = kPacked ? p.Hkv : (int)gridDim.x;
  const int n_tiles = (L + kTile - 1) / kTile;
  const int i_start = p.causal ? jt : 0;
  const int n_i = n_tiles - i_start;
  // Steps t_begin .. t_begin + n_steps - 1 of the key tile's G * n_i (query head, query tile)
  // steps; the loops below count t from 0, step t being the key tile's step t_begin + t.
  const int t_begin = (int)((long long)sp.part * (G * n_i) / sp.parts);
  const int n_steps = (int)((long long)(sp.part + 1) * (G * n_i) / sp.parts) - t_begin;
  // D / LSE2 rows of query tile i of query head bhq0 + hl: copied from the 16-byte aligned row
  // below (the copy is 4 rows wider when a packed sequence starts off a multiple of 4 rows).
  constexpr int n_rowfl = kPacked ? kTile + 4 : kTile;
  auto rows_at = [&](int hl, int i) { return (size_t)(bhq0 + hl) * p.S_pad + (size_t)row0 + (size_t)i * kTile; };
  const WaitGuard wg{&bars->abort_flag, p.status, kWaitLimitNs};

  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->do_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);   // the reduce warp, once its dQ reduces have read the stage
      mbar_init(&bars->do_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 8);   // one arrival per element-wise warp
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 8);
    mbar_init(&bars->stage_full, 8);
    mbar_init(&bars->dkv_done, 1);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->k_ready, 8);
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
  // Q(t) and step t's -LSE2 / D rows into stage t % ST, on q_full (one thread).
  auto load_q_rows = [&](int t) {
    const int st = t % ST;
    const int hl = (t_begin + t) / n_i;
    const int i = i_start + (t_begin + t - hl * n_i);
    const int bhq = bhq0 + hl;
    uint64_t* bar = &bars->q_full[st];
    mbar_arrive_expect_tx(bar, C::kTileBytes + 2 * n_rowfl * 4);
    for (int c = 0; c < C::kChunks; ++c) {
      const bool q_ok = dbg_tile(c * kChunk, row0 + i * kTile, bhq, D, kChunk, row0, row0 + L, heads_q, p.status);
      tma_load_3d_chk(smem + C::kQOff + st * C::kTileBytes + c * kBoxBytes, &map_q, bar, c * kChunk, row0 + i * kTile,
                      bhq, q_ok);
    }
    float* srow = reinterpret_cast<float*>(smem + C::kRowOff) + st * 2 * C::kRowFl;
    const size_t roff = rows_at(hl, i) & ~size_t(3);
    if (dbg_range((long long)roff, n_rowfl, p.rows_total, p.status)) {
      bulk_load(srow, p.nlse2 + roff, n_rowfl * 4, bar);
      bulk_load(srow + C::kRowFl, p.dvec + roff, n_rowfl * 4, bar);
    } else {
      mbar_complete_tx(bar, 2 * n_rowfl * 4);
    }
  };

  // dO(t) into stage t % ST, on do_full (one thread).
  auto load_do = [&](int t) {
    const int st = t % ST;
    const int hl = (t_begin + t) / n_i;
    const int i = i_start + (t_begin + t - hl * n_i);
    const int bhq = bhq0 + hl;
    uint64_t* bar = &bars->do_full[st];
    mbar_arrive_expect_tx(bar, C::kTileBytes);
    for (int c = 0; c < C::kChunks; ++c) {
      const bool q_ok = dbg_tile(c * kChunk, row0 + i * kTile, bhq, D, kChunk, row0, row0 + L, heads_q, p.status);
      tma_load_3d_chk(smem + C::kDOOff + st * C::kTileBytes + c * kBoxBytes, &map_do, bar, c * kChunk,
                      row0 + i * kTile, bhq, q_ok);
    }
  };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      tma_prefetch_desc(&map_do);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        const bool kv_ok =
            dbg_tile(c * kChunk, row0 + jt * kTile, kv_coord, D, kChunk, row0, row0 + L, heads_kv, p.status);
        tma_load_3d_chk(smem + C::kKOff + c * kBoxBytes, &map_k, &bars->kv_full, c * kChunk, row0 + jt * kTile,
                        kv_coord, kv_ok);
        tma_load_3d_chk(smem + C::kVOff + c * kBoxBytes, &map_v, &bars->kv_full, c * kChunk, row0 + jt * kTile,
                        kv_coord, kv_ok);
      }
      int issued = 0, issued_do = 0;
      // Q(t) with its rows, then dO(t). With the dQ partials only the first ST steps' tiles come
      // from here: for later steps the reduce warp loads them into a stage as soon as it has read
      // the half of the partial staged there, so that the loads do not share the TMA unit with
      // the other half's reduce-adds.
      const int n_own = kDq ? (n_steps < ST ? n_steps : ST) : n_steps;
      for (int t = 0; t < n_own; ++t) {
        const int st = t % ST;
        const int use = t / ST;
        if (use > 0 && !mbar_wait(&bars->q_empty[st], (use - 1) & 1, wg)) break;
        load_q_rows(t);
        issued = t + 1;
        if (use > 0 && !mbar_wait(&bars->do_empty[st], (use - 1) & 1, wg)) break;
        load_do(t);
        issued_do = t + 1;
      }
      if (bars->abort_flag) {
        mbar_wait_drain(&bars->kv_full, 0, kWaitLimitNs);
        for (int t = (issued > ST ? issued - ST : 0); t < issued; ++t)
          mbar_wait_drain(&bars->q_full[t % ST], (t / ST) & 1, kWaitLimitNs);
        for (int t = (issued_do > ST ? issued_do - ST : 0); t < issued_do; ++t)
          mbar_wait_drain(&bars->do_full[t % ST], (t / ST) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_kk = idesc_bf16(128, 128, false, false);  // S^T, dP^T: both operands K-major
      constexpr uint32_t idesc_tb = idesc_bf16(128, D, false, true);     // dV, dK: A in TMEM, B MN-major
      constexpr uint32_t idesc_mm = idesc_bf16(128, D, true, true);      // dQ: A and B MN-major
      // Descriptors are built once; an MMA only adds a compile-time offset (the start-address field
      // is the low 14 bits of the descriptor and never carries).
      constexpr uint64_t kTileDesc = (uint64_t)(C::kTileBytes >> 4);
      const uint64_t dk_k = sdesc_sw128(smem_addr(smem + C::kKOff), 16, 1024);          // K as K-major A
      const uint64_t dv_k = sdesc_sw128(smem_addr(smem + C::kVOff), 16, 1024);          // V as K-major A
      const uint64_t dk_mn = sdesc_sw128(smem_addr(smem + C::kKOff), kBoxBytes, 1024);  // K as MN-major B
      const uint64_t dq_k0 = sdesc_sw128(smem_addr(smem + C::kQOff), 16, 1024);
      const uint64_t dq_mn0 = sdesc_sw128(smem_addr(smem + C::kQOff), kBoxBytes, 1024);
      const uint64_t ddo_k0 = sdesc_sw128(smem_addr(smem + C::kDOOff), 16, 1024);
      const uint64_t ddo_mn0 = sdesc_sw128(smem_addr(smem + C::kDOOff), kBoxBytes, 1024);
      const uint64_t dds_mn = sdesc_sw128(smem_addr(smem + C::kDSOff), kBoxBytes, 1024);
      // X^T = A B^T for a 128-row A tile (K or V) and a 128-row B tile (Q or dO), both K-major.
      auto issue_kmajor = [=](uint32_t d_col, uint64_t a, uint64_t bb) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
          umma_ss(tbase + d_col, a + off, bb + off, idesc_kk, kk > 0 ? 1u : 0u);
        }
      };
      auto stage_desc = [=](uint64_t base, int t) { return base + (uint64_t)(t % ST) * kTileDesc; };
      // TMEM column of the A operand (P^T; dS^T is 32 columns further) for query rows 16kk..16kk+15:
      // column half h = kk / 4 keeps its packed P^T in [64h, 64h+32) and dS^T in [64h+32, 64h+64).
      auto p_col = [](int kk) { return (uint32_t)(kk >> 2) * 64u + (uint32_t)(kk & 3) * 8u; };
      bool ok = mbar_wait(&bars->kv_full, 0, wg) && mbar_wait(&bars->q_full[0], 0, wg);
      if (kRope && ok) ok = mbar_wait(&bars->k_ready, 0, wg);  // keys rotated by the element-wise warps
      if (ok) {
        tc_fence_after();
        issue_kmajor(C::kSPCol, dk_k, stage_desc(dq_k0, 0));
        umma_commit(&bars->s_full);
      }
      if (ok) ok = mbar_wait(&bars->do_full[0], 0, wg);
      if (ok) {
        tc_fence_after();
        issue_kmajor(C::kDPCol, dv_k, stage_desc(ddo_k0, 0));
        umma_commit(&bars->dp_full);
      }
      for (int t = 0; ok && t < n_steps; ++t) {
        if (!(ok = mbar_wait(&bars->p_full, t & 1, wg))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts(tbase + C::kDVCol, tbase + C::kSPCol + p_col(kk),
                  stage_desc(ddo_mn0, t) + (uint64_t)((kk * 2048) >> 4), idesc_tb, (t > 0 || kk > 0) ? 1u : 0u);
        if (!(ok = mbar_wait(&bars->ds_full, t & 1, wg))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts(tbase + C::kDKCol, tbase + C::kSPCol + p_col(kk) + 32u,
                  stage_desc(dq_mn0, t) + (uint64_t)((kk * 2048) >> 4), idesc_tb, (t > 0 || kk > 0) ? 1u : 0u);
        if (kDq) {
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_ss(tbase + C::kDPCol, dds_mn + (uint64_t)((kk * 2048) >> 4), dk_mn + (uint64_t)((kk * 2048) >> 4),
                    idesc_mm, kk > 0 ? 1u : 0u);
          umma_commit(&bars->dq_full);
        } else {
          umma_commit(&bars->q_empty[t % ST]);  // dK(t) and dV(t) were the last readers of Q(t), dO(t)
          umma_commit(&bars->do_empty[t % ST]);
        }
        if (t + 1 < n_steps) {
          const int t1 = t + 1;
          if (!(ok = mbar_wait(&bars->q_full[t1 % ST], (t1 / ST) & 1, wg))) break;
          tc_fence_after();
          issue_kmajor(C::kSPCol, dk_k, stage_desc(dq_k0, t1));  // P^T(t), dS^T(t) were consumed by dV(t), dK(t)
          umma_commit(&bars->s_full);
          if (kDq) {  // dP(t+1) overwrites the dQ(t) partial: wait until it has been read out
            if (!(ok = mbar_wait(&bars->dq_free, t & 1, wg))) break;
          }
          if (!(ok = mbar_wait(&bars->do_full[t1 % ST], (t1 / ST) & 1, wg))) break;
          tc_fence_after();
          issue_kmajor(C::kDPCol, dv_k, stage_desc(ddo_k0, t1));
          umma_commit(&bars->dp_full);
        }
      }
      umma_commit(&bars->dkv_done);
      umma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, kWaitLimitNs);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ dQ reduce warp
    // Issues the TMA reduce-adds of each step's staged dQ partial; once the half staged in the
    // step's Q tile has been read it loads Q(t + ST) into that stage, and once the dO half has
    // been read it hands the dO stage back to the producer.
    if (kDq && lane == 0) {
      tma_prefetch_desc(&map_acc);
      tma_prefetch_desc(&map_q);
      int q_issued = ST < n_steps ? ST : n_steps;  // Q(0 .. ST-1) come from the producer
      for (int t = 0; t < n_steps; ++t) {
        if (!mbar_wait(&bars->stage_full, t & 1, wg)) break;
        const int st = t % ST;
        const int hl = (t_begin + t) / n_i;
        const int i = i_start + (t_begin + t - hl * n_i);
        const int bhq = bhq0 + hl;
        // The slices staged in the Q tile go first, in their own bulk group; once they have been
        // read, this thread loads Q(t + ST) into the stage itself, before it issues the slices
        // staged in the dO tile, so that the load does not share the TMA unit with them.
#pragma unroll
        for (int s2 = 0; s2 < C::kChunks; ++s2)
          if (dbg_tile(s2 * 32, row0 + i * kTile, bhq, D, 32, row0, row0 + L, heads_q, p.status))
            tma_reduce_add_3d(&map_acc, smem + C::kQOff + st * C::kTileBytes + s2 * kBoxBytes, s2 * 32,
                              row0 + i * kTile, bhq);
        bulk_commit_group();
        bulk_wait_group_read<0>();
        if (t + ST < n_steps) {
          load_q_rows(t + ST);
          q_issued = t + ST + 1;
        }
#pragma unroll
        for (int s2 = C::kChunks; s2 < D / 32; ++s2)
          if (dbg_tile(s2 * 32, row0 + i * kTile, bhq, D, 32, row0, row0 + L, heads_q, p.status))
            tma_reduce_add_3d(&map_acc, smem + C::kDOOff + st * C::kTileBytes + (s2 - C::kChunks) * kBoxBytes,
                              s2 * 32, row0 + i * kTile, bhq);
        bulk_commit_group();
        bulk_wait_group_read<0>();
        if (t + ST < n_steps) load_do(t + ST);
      }
      bulk_wait_group<0>();
      if (bars->abort_flag) {  // let the Q and dO loads this thread issued land
        for (int tt = (q_issued - ST > ST ? q_issued - ST : ST); tt < q_issued; ++tt) {
          mbar_wait_drain(&bars->q_full[tt % ST], (tt / ST) & 1, kWaitLimitNs);
          mbar_wait_drain(&bars->do_full[tt % ST], (tt / ST) & 1, kWaitLimitNs);
        }
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ element-wise warps 0..7
    const int quarter = warp & 3;
    const int hf = warp >> 2;                     // column half
    const int row = quarter * 32 + lane;          // TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t sp_tmem = tbase + lane_off + C::kSPCol;
    const uint32_t dp_tmem = tbase + lane_off + C::kDPCol;
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    const int kv_row = jt * kTile + row;
    const bool kv_valid = kv_row < L;
    uint8_t* sds_half = smem + C::kDSOff + hf * kBoxBytes;  // dS columns [64hf, 64hf+64)
    bool ok = true;
    if (kRope) {
      // Rotary embedding: thread (row, hf) turns half of its key row's pairs in shared memory.
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->kv_full, 0, wg));
      if (ok && kv_valid && dbg_range((long long)(row0 + kv_row) * (D / 2), D / 2, (long long)p.S * (D / 2), p.status)) {
        const int pos = row0 + kv_row;  // position within the (dense) sequence
        rope_rotate_row_smem<D>(smem + C::kKOff, row, p.rope_cos + (size_t)pos * (D / 2),
                                p.rope_sin + (size_t)pos * (D / 2), 1.f, hf * (D / 32), (hf + 1) * (D / 32));
      }
      fence_proxy_async_smem();
      mbar_arrive_warp(&bars->k_ready);
    }
    for (int t = 0; t < n_steps; ++t) {
      const int st = t % ST;
      const int hl = (t_begin + t) / n_i;
      const int i = i_start + (t_begin + t - hl * n_i);
      const int roff = kPacked ? (int)(rows_at(hl, i) & 3) : 0;  // the rows' offset within their widened copy
      const float* snl = reinterpret_cast<const float*>(smem + C::kRowOff) + st * 2 * C::kRowFl + roff + hf * 64;
      const float* sdv = snl + C::kRowFl;
      // visible iff key (jt*128 + row) <= query (i*128 + col): on the diagonal tile, col >= row
      const int first_visible = (p.causal && i == jt) ? row : 0;
      // Packed: query columns at or past q_limit lie beyond the sequence (dense: -LSE2 = -inf there).
      const int q_limit = kPacked ? L - i * kTile : kTile;

      // ---- P^T = exp2(S^T c - LSE2) for the 64 query columns of this half
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full, t & 1, wg));
      if (!ok) break;
      tc_fence_after();
      float P[64];
      {
        uint32_t r[64];
        tmem_ld_32x32b_x32(sp_tmem + hf * 64, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld_32x32b_x32(sp_tmem + hf * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        uint32_t pk[32];
        // causal diagonal, keys past the sequence, or queries past it
        const bool masked = first_visible > hf * 64 || !kv_valid || (kPacked && q_limit < hf * 64 + 64);
        if (masked) {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int c0 = 2 * x;
            const int col = hf * 64 + c0;
            const float2 a = ffma2(make_float2(__uint_as_float(r[c0]), __uint_as_float(r[c0 + 1])), c2,
                                   make_float2(snl[c0], snl[c0 + 1]));
            const float e0 = ex2_approx(a.x);
            const float e1 = ex2_approx(a.y);
            P[c0] = (kv_valid && col >= first_visible && col < q_limit) ? e0 : 0.f;
            P[c0 + 1] = (kv_valid && col + 1 >= first_visible && col + 1 < q_limit) ? e1 : 0.f;
            pk[x] = pack_bf16(P[c0], P[c0 + 1]);
          }
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int c0 = 2 * x;
            const float2 a = ffma2(make_float2(__uint_as_float(r[c0]), __uint_as_float(r[c0 + 1])), c2,
                                   make_float2(snl[c0], snl[c0 + 1]));
            P[c0] = ex2_approx(a.x);
            P[c0 + 1] = ex2_approx(a.y);
            pk[x] = pack_bf16(P[c0], P[c0 + 1]);
          }
        }
        tmem_st_32x32b_x32(sp_tmem + hf * 64, pk);  // this half's own columns
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&bars->p_full);

      // ---- dS^T = P^T (dP^T - D): into TMEM (A operand of dK) and into smem (A operand of dQ)
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->dp_full, t & 1, wg));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t d[32];
        tmem_ld_32x32b_x32(dp_tmem + hf * 64 + q * 32, d);
        tmem_wait_ld_x32(d);
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int c0 = q * 32 + 2 * x;
          const float2 ds = fmul2(make_float2(P[c0], P[c0 + 1]),
                                  fsub2(make_float2(__uint_as_float(d[2 * x]), __uint_as_float(d[2 * x + 1])),
                                        make_float2(sdv[c0], sdv[c0 + 1])));
          pk[x] = pack_bf16(ds.x, ds.y);
        }
        tmem_st_32x32b_x16(sp_tmem + hf * 64 + 32 + q * 16, pk);
        // dS[row = key][col = query] into the MN-major (query-contiguous) 128B-swizzled tile.
        if (kDq) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int unit = q * 4 + u;  // 16-byte unit within this half's 128-byte row
            *reinterpret_cast<uint4*>(sds_half + (row >> 3) * 1024 + (row & 7) * 128 + ((unit ^ (row & 7)) << 4)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        }
      }
      if (kDq) fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&bars->ds_full);
      if (!kDq) continue;

      ok = __all_sync(0xffffffffu, mbar_wait(&bars->dq_full, t & 1, wg));
      if (!ok) break;
      tc_fence_after();
      // ---- dQ partial (TMEM lane = query row): load this half's columns, free TMEM, stage it
      uint32_t dq[C::kRounds][32];
#pragma unroll
      for (int rd = 0; rd < C::kRounds; ++rd) tmem_ld_32x32b_x32(dp_tmem + (2 * rd + hf) * 32, dq[rd]);
#pragma unroll
      for (int rd = 0; rd < C::kRounds; ++rd) tmem_wait_ld_x32(dq[rd]);
      tc_fence_before();
      mbar_arrive_warp(&bars->dq_free);
      // Staging, all slices at once, into this step's Q and dO tiles (their last readers, dK(t)
      // and dV(t), completed before dQ(t)): slice 2rd + hf goes to box 2rd + hf of [Q boxes,
      // dO boxes]; the reduce warp sends them on.
#pragma unroll
      for (int rd = 0; rd < C::kRounds; ++rd) {
        const int box = 2 * rd + hf;
        float* stage = reinterpret_cast<float*>(
            box < C::kChunks ? smem + C::kQOff + st * C::kTileBytes + box * kBoxBytes
                             : smem + C::kDOOff + st * C::kTileBytes + (box - C::kChunks) * kBoxBytes);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<float4*>(stage + row * 32 + ((u ^ (row & 7)) << 2)) =
              make_float4(__uint_as_float(dq[rd][4 * u]), __uint_as_float(dq[rd][4 * u + 1]),
                          __uint_as_float(dq[rd][4 * u + 2]), __uint_as_float(dq[rd][4 * u + 3]));
      }
      fence_proxy_async_smem();
      mbar_arrive_warp(&bars->stage_full);
      if (!ok) break;
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->dkv_done, 0, wg));
    if (kRope && ok) {
      // dK of the unrotated keys: thread (row, hf) takes pairs [hf D/4, hf D/4 + D/4), i.e. its
      // columns c and c + D/2, and turns them back by the transposed rotation.
      tc_fence_after();
      constexpr int kQ = D / 4;
      const int i0 = hf * kQ;
      uint32_t lo[kQ], hi[kQ];
      if constexpr (D == 128) {
        tmem_ld_32x32b_x32(tbase + lane_off + C::kDKCol + i0, lo);
        tmem_ld_32x32b_x32(tbase + lane_off + C::kDKCol + D / 2 + i0, hi);
        tmem_wait_ld_x32(lo);
        tmem_wait_ld_x32(hi);
      } else {
        tmem_ld_32x32b_x16(tbase + lane_off + C::kDKCol + i0, lo);
        tmem_ld_32x32b_x16(tbase + lane_off + C::kDKCol + D / 2 + i0, hi);
        tmem_wait_ld_x16(lo);
        tmem_wait_ld_x16(hi);
      }
      if (kv_valid && dbg_range(((long long)kv_coord * p.S + row0 + kv_row) * D, D, (long long)heads_kv * p.S * D,
                                p.status) &&
          dbg_range((long long)(row0 + kv_row) * (D / 2), D / 2, (long long)p.S * (D / 2), p.status)) {
        const int pos = row0 + kv_row;
        const float* cs = p.rope_cos + (size_t)pos * (D / 2) + i0;
        const float* sn = p.rope_sin + (size_t)pos * (D / 2) + i0;
        uint16_t* dst = p.dk + ((size_t)kv_coord * p.S + row0 + kv_row) * D;
        const float sc = p.scale;
#pragma unroll
        for (int x = 0; x < kQ / 8; ++x) {
          uint32_t wl[4], wh[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int i = 8 * x + 2 * w;
            const float a0 = __uint_as_float(lo[i]) * sc, a1 = __uint_as_float(lo[i + 1]) * sc;
            const float b0 = __uint_as_float(hi[i]) * sc, b1 = __uint_as_float(hi[i + 1]) * sc;
            const float c0 = __ldg(cs + i), c1 = __ldg(cs + i + 1), s0 = __ldg(sn + i), s1 = __ldg(sn + i + 1);
            wl[w] = pack_bf16(a0 * c0 + b0 * s0, a1 * c1 + b1 * s1);
            wh[w] = pack_bf16(b0 * c0 - a0 * s0, b1 * c1 - a1 * s1);
          }
          *reinterpret_cast<uint4*>(dst + i0 + 8 * x) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
          *reinterpret_cast<uint4*>(dst + D / 2 + i0 + 8 * x) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        }
      }
    }
    if (ok && sp.parts > 1) {
      // Split key tile: this part's f32 dK (unscaled) and dV go to its partial slot; the part that
      // takes the last ticket adds all parts in part order and writes dK, dV.
      tc_fence_after();
      constexpr size_t kSlot = (size_t)kTile * D * 2;  // a partial: dV [128][D], then dK [128][D]
      float* slots = p.part + ((size_t)grp * p.parts_per_group + sp.pidx) * kSlot;
      const size_t slot_end = (size_t)gridDim.x * p.parts_per_group * kSlot;  // the partials' extent
#pragma unroll
      for (int q = 0; q < D / 64; ++q) {
        const int col = hf * (D / 2) + q * 32;
        uint32_t dv[32], dk[32];
        tmem_ld_32x32b_x32(tbase + lane_off + C::kDVCol + col, dv);
        tmem_ld_32x32b_x32(tbase + lane_off + C::kDKCol + col, dk);
        tmem_wait_ld_x32(dv);
        tmem_wait_ld_x32(dk);
        const size_t at = (size_t)sp.part * kSlot + (size_t)row * D + col;
        if (kv_valid &&
            dbg_range((long long)(slots - p.part) + (long long)at, (long long)kTile * D + 32, (long long)slot_end,
                      p.status) &&
            dbg_ok((reinterpret_cast<uintptr_t>(slots + at) & 15u) == 0, p.status)) {
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            *reinterpret_cast<float4*>(slots + at + 4 * x) =
                make_float4(__uint_as_float(dv[4 * x]), __uint_as_float(dv[4 * x + 1]), __uint_as_float(dv[4 * x + 2]),
                            __uint_as_float(dv[4 * x + 3]));
            *reinterpret_cast<float4*>(slots + at + (size_t)kTile * D + 4 * x) =
                make_float4(__uint_as_float(dk[4 * x]), __uint_as_float(dk[4 * x + 1]), __uint_as_float(dk[4 * x + 2]),
                            __uint_as_float(dk[4 * x + 3]));
          }
        }
      }
      // Every element-wise thread's partial stores precede thread 0's fence and ticket (the barrier
      // orders them within the CTA, the fence is cumulative); the last part's fence after its ticket
      // orders the other parts' stores before the reads that follow the second barrier.
      uint32_t ephase = 0;
      ok = wg_barrier(&bars->epi_bar, ephase, wg);
      if (ok && tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(p.tickets + (size_t)grp * p.n_ktiles + jt, 1u);
        bars->last = (prev == (unsigned)sp.parts - 1u) ? 1 : 0;
        __threadfence();
      }
      if (ok) ok = wg_barrier(&bars->epi_bar, ephase, wg);
      if (ok && bars->last && kv_valid) {
        const size_t orow = ((size_t)kv_coord * p.S + row0 + kv_row) * D;
#pragma unroll
        for (int q = 0; q < D / 64; ++q) {
          const int col = hf * (D / 2) + q * 32;
          float sv[32], sk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) sv[e] = sk[e] = 0.f;
          for (int pp = 0; pp < sp.parts; ++pp) {  // part order, whichever part arrived last
            const float* src = slots + (size_t)pp * kSlot + (size_t)row * D + col;
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              const float4 a = __ldcg(reinterpret_cast<const float4*>(src) + x);
              const float4 b = __ldcg(reinterpret_cast<const float4*>(src + (size_t)kTile * D) + x);
              sv[4 * x] += a.x; sv[4 * x + 1] += a.y; sv[4 * x + 2] += a.z; sv[4 * x + 3] += a.w;
              sk[4 * x] += b.x; sk[4 * x + 1] += b.y; sk[4 * x + 2] += b.z; sk[4 * x + 3] += b.w;
            }
          }
          if (dbg_range((long long)orow + col, 32, (long long)heads_kv * p.S * D, p.status)) {
            uint4* dstv = reinterpret_cast<uint4*>(p.dv + orow + col);
            uint4* dstk = reinterpret_cast<uint4*>(p.dk + orow + col);
            const float sc = p.scale;
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              dstv[x] = make_uint4(pack_bf16(sv[8 * x], sv[8 * x + 1]), pack_bf16(sv[8 * x + 2], sv[8 * x + 3]),
                                   pack_bf16(sv[8 * x + 4], sv[8 * x + 5]), pack_bf16(sv[8 * x + 6], sv[8 * x + 7]));
              dstk[x] = make_uint4(pack_bf16(sk[8 * x] * sc, sk[8 * x + 1] * sc),
                                   pack_bf16(sk[8 * x + 2] * sc, sk[8 * x + 3] * sc),
                                   pack_bf16(sk[8 * x + 4] * sc, sk[8 * x + 5] * sc),
                                   pack_bf16(sk[8 * x + 6] * sc, sk[8 * x + 7] * sc));
            }
          }
        }
      }
    } else if (ok) {
      tc_fence_after();
      const size_t orow = ((size_t)kv_coord * p.S + row0 + kv_row) * D;
#pragma unroll
      for (int q = 0; q < D / 64; ++q) {
        const int col = hf * (D / 2) + q * 32;
        uint32_t dv[32], dk[32];
        tmem_ld_32x32b_x32(tbase + lane_off + C::kDVCol + col, dv);
        tmem_ld_32x32b_x32(tbase + lane_off + C::kDKCol + col, dk);
        tmem_wait_ld_x32(dv);
        tmem_wait_ld_x32(dk);
        if (kv_valid && dbg_range((long long)orow + col, 32, (long long)heads_kv * p.S * D, p.status)) {
          uint4* dstv = reinterpret_cast<uint4*>(p.dv + orow + col);
          uint4* dstk = reinterpret_cast<uint4*>(p.dk + orow + col);
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            dstv[x] = make_uint4(pack_bf16(__uint_as_float(dv[8 * x + 0]), __uint_as_float(dv[8 * x + 1])),
                                 pack_bf16(__uint_as_float(dv[8 * x + 2]), __uint_as_float(dv[8 * x + 3])),
                                 pack_bf16(__uint_as_float(dv[8 * x + 4]), __uint_as_float(dv[8 * x + 5])),
                                 pack_bf16(__uint_as_float(dv[8 * x + 6]), __uint_as_float(dv[8 * x + 7])));
            const float s = p.scale;
            if (!kRope) {  // with the rotary embedding dK was stored, turned back, above
              dstk[x] = make_uint4(pack_bf16(__uint_as_float(dk[8 * x + 0]) * s, __uint_as_float(dk[8 * x + 1]) * s),
                                   pack_bf16(__uint_as_float(dk[8 * x + 2]) * s, __uint_as_float(dk[8 * x + 3]) * s),
                                   pack_bf16(__uint_as_float(dk[8 * x + 4]) * s, __uint_as_float(dk[8 * x + 5]) * s),
                                   pack_bf16(__uint_as_float(dk[8 * x + 6]) * s, __uint_as_float(dk[8 * x + 7]) * s));
            }
          }
        }
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

// Plan selection for the split backward. The time of a CTA is modelled as its steps plus a fixed
// cost of kCtaOverheadSteps steps (prologue, epilogue, partials; measured on GB300 at D = 64: a
// 16-step CTA takes ~43 us, two 4-step CTAs in a row ~34 us), CTAs are dealt longest first onto
// kPlanCtas SMs (the order of the grid), and the cap with the shortest estimated makespan wins if
// it beats the unsplit grid by kSplitGain. Only grids of at most two waves are considered.
constexpr int kCtaOverheadSteps = 4;
constexpr double kSplitGain = 1.15;

long long bwd_plan_makespan(int B, int Hkv, int G, int n_tiles, int causal, int cap) {
  std::vector<int> sizes;
  for (int jt = 0; jt < n_tiles; ++jt) {
    const int steps = bwd_tile_steps(jt, n_tiles, G, causal);
    const int parts = cap > 0 ? ceil_div(steps, cap) : 1;
    for (int pp = 0; pp < parts; ++pp) {
      const int sz = (int)((long long)(pp + 1) * steps / parts - (long long)pp * steps / parts);
      for (int g = 0; g < B * Hkv; ++g) sizes.push_back(sz + kCtaOverheadSteps);
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
  return span;
}

BwdSplit bwd_split_plan_uncached(int B, int Hkv, int G, int n_tiles, int causal) {
  BwdSplit sp{0, n_tiles, 0};
  const int steps0 = bwd_tile_steps(0, n_tiles, G, causal);
  if ((long long)B * Hkv * n_tiles > 2ll * kPlanCtas || steps0 < 2) return sp;
  const long long unsplit = bwd_plan_makespan(B, Hkv, G, n_tiles, causal, 0);
  long long best = unsplit;
  int best_cap = 0;
  for (int cap = steps0 - 1; cap >= 1; --cap) {
    // Grids of more than four waves are not considered; smaller caps only add CTAs, so the
    // search (and its host time on a first call) stops there.
    long long ctas = 0;
    for (int jt = 0; jt < n_tiles; ++jt) ctas += ceil_div(bwd_tile_steps(jt, n_tiles, G, causal), cap);
    if ((long long)B * Hkv * ctas > 4ll * kPlanCtas) break;
    const long long m = bwd_plan_makespan(B, Hkv, G, n_tiles, causal, cap);
    if (m < best) {
      best = m;
      best_cap = cap;
    }
  }
  if (best_cap == 0 || (double)best * kSplitGain > (double)unsplit) return sp;
  sp.cap = best_cap;
  sp.ctas_per_group = 0;
  for (int jt = 0; jt < n_tiles; ++jt) {
    const int parts = ceil_div(bwd_tile_steps(jt, n_tiles, G, causal), sp.cap);
    sp.ctas_per_group += parts;
    if (parts > 1) sp.parts_per_group += parts;
  }
  return sp;
}

}  // namespace

BwdSplit bwd_split_plan(int B, int Hkv, int G, int n_tiles, int causal) {
  struct Entry {
    int key[5];
    BwdSplit plan;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  const int key[5] = {B, Hkv, G, n_tiles, causal ? 1 : 0};
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry& e : cache)
      if (std::equal(key, key + 5, e.key)) return e.plan;
  }
  const BwdSplit plan = bwd_split_plan_uncached(B, Hkv, G, n_tiles, causal);
  std::lock_guard<std::mutex> lk(mu);
  if (cache.size() < 256) cache.push_back(Entry{{key[0], key[1], key[2], key[3], key[4]}, plan});
  return plan;
}

namespace {

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const bool det = a.deterministic != 0;  // dQ by the query-major kernel, no f32 accumulator
  const bool packed = a.cu != nullptr;
  const int n_tiles = ceil_div(packed ? a.max_seqlen : a.S, kTile);  // key tiles of the longest sequence
  const int S_pad = packed ? a.S : ceil_div(a.S, kTile) * kTile;     // row stride of D / LSE2
  const int rows_valid = packed ? a.Hq * a.S : a.B * a.Hq * S_pad;
  const int rows_total = packed ? rows_valid + kRowPad : rows_valid;
  const long long acc_elems = det ? 0 : (long long)(packed ? 1 : a.B) * a.Hq * a.S * D;
  const int sms = device_sm_count();
  // A small dense problem has its heaviest key tiles split across CTAs (BwdSplit); the rotary
  // variant, which turns dK back in the epilogue, and packed batches are not split.
  const BwdSplit split = (!packed && !a.rope_cos) ? bwd_split_plan(a.B, a.Hkv, a.Hq / a.Hkv, n_tiles, a.causal)
                                                  : BwdSplit{0, n_tiles, 0};
  const int n_tickets = split.cap > 0 ? a.B * a.Hkv * n_tiles : 0;
  {
    const int threads = 256;
    long long want = ((long long)rows_total * (D / 8) + threads - 1) / threads;
    const int blocks = (int)(want < (long long)sms * 8 ? (want < 1 ? 1 : want) : (long long)sms * 8);
    trace_begin(kKernelBwdPrep, stream);
    cudaError_t e = launch_pdl(bwd_prep_kernel<D>, dim3(blocks), dim3(threads), 0, stream,
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dO), a.lse, a.dvec, a.nlse2, a.dq_acc,
        rows_total, rows_valid, a.S, S_pad, 1.4426950408889634f, acc_elems / 4, a.tickets, n_tickets, a.status);
    if (e == cudaSuccess) e = cudaGetLastError();
    trace_end(kKernelBwdPrep, stream);
    if (e != cudaSuccess) return e;
  }
  {
    BwdKParams p;
    p.nlse2 = a.nlse2;
    p.dvec = a.dvec;
    p.dk = static_cast<uint16_t*>(a.dk);
    p.dv = static_cast<uint16_t*>(a.dv);
    p.cu = a.cu;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.S = a.S;
    p.S_pad = S_pad;
    p.causal = a.causal;
    p.max_seqlen = a.max_seqlen;
    p.n_ktiles = n_tiles;
    p.rows_total = rows_total;
    p.cap = split.cap;
    p.ctas_per_group = split.ctas_per_group;
    p.parts_per_group = split.parts_per_group;
    p.part = a.part;
    p.tickets = a.tickets;
    p.rope_cos = a.rope_cos;
    p.rope_sin = a.rope_sin;
    p.scale = a.scale;
    p.scale_log2 = a.scale_log2;
    p.status = a.status;
    auto kern = packed ? bwd_main_kernel<D, true, false, true>
                : det ? bwd_main_kernel<D, false, false, false>
                      : (a.rope_cos ? bwd_main_kernel<D, true, true, false> : bwd_main_kernel<D, true, false, false>);
    const KernelKind kind = det ? kKernelBwdDkdv : kKernelBwdMain;
    cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads, 0);
    if (e != cudaSuccess) return e;
    const long long packed_ctas = (long long)a.B * a.Hkv * n_tiles;
    if (packed && packed_ctas >= (1ll << 31)) return cudaErrorInvalidValue;
    const dim3 grid = packed ? dim3((unsigned)packed_ctas)
                             : dim3((unsigned)(a.B * a.Hkv), (unsigned)(split.cap > 0 ? split.ctas_per_group : n_tiles));
    trace_begin(kind, stream);
    e = launch_pdl(kern, grid, dim3(C::kThreads), C::kSmemBytes, stream, *a.map_q, *a.map_k, *a.map_v, *a.map_do,
                   *a.map_dqacc, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    trace_end(kind, stream);
    if (e != cudaSuccess) return e;
  }
  if (det) return launch_bwd_dq(a, stream);
  if (a.rope_cos)  // dQ of the unrotated queries
    return launch_rope_convert(a.dq_acc, a.dq, a.rope_cos, a.rope_sin, (long long)a.B * a.Hq * a.S, a.S, D, a.scale,
                               a.status, stream);
  {
    const long long n8 = acc_elems / 8;
    const int threads = 256;
    long long want = (n8 + threads - 1) / threads;
    const int blocks = (int)(want < (long long)sms * 8 ? (want < 1 ? 1 : want) : (long long)sms * 8);
    trace_begin(kKernelBwdConvert, stream);
    cudaError_t e = launch_pdl(bwd_convert_kernel, dim3(blocks), dim3(threads), 0, stream, a.dq_acc,
                               static_cast<uint16_t*>(a.dq), n8, a.scale);
    if (e == cudaSuccess) e = cudaGetLastError();
    trace_end(kKernelBwdConvert, stream);
    return e;
  }
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  if (a.D == 64) return launch_bwd_d<64>(a, stream);
  return launch_bwd_d<128>(a, stream);
}

}  // namespace gqa
