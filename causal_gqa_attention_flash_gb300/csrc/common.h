// Definitions shared by the kernels and the host-side launchers of libgqa_attn.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace gqa {

// Tile edge along the sequence for queries and keys (one tcgen05 M=128 tile).
constexpr int kTile = 128;
// Columns of one 128-byte swizzle row of bf16 (the TMA box's inner extent).
constexpr int kChunk = 64;
// Bytes of one [128 rows x 64 bf16] swizzled box.
constexpr int kBoxBytes = kTile * kChunk * 2;

// Time limit of one device-side wait before the kernel gives up (ns).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Launch with programmatic stream serialization: the kernel may be scheduled while the kernel
// ahead of it in the stream finishes, hiding the launch gap between them. Every kernel launched
// this way calls griddep_wait() before anything else, so it reads nothing before its
// predecessor has completed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct FwdArgs {
  const CUtensorMap* map_q;  // [B*Hq, Sq, D] bf16, box {64, 128, 1}, 128B swizzle
  const CUtensorMap* map_k;  // [B*Hkv, Sk, D]
  const CUtensorMap* map_v;
  const CUtensorMap* map_o;  // [B*Hq, Sq, D] bf16 (TMA store of O)
  float* lse;                // f32 [B, Hq, Sq]
  void* o;                   // O itself (packed batches store ragged tiles row by row)
  const int* cu_q;           // packed batch: device int32 [B + 1] query bounds; nullptr = dense
  const int* cu_k;           // packed batch: key bounds
  int max_seqlen_q;          // packed batch: bound on every sequence's query count
  const float* rope_cos;     // rotary tables f32 [S, D/2] (nullptr: no rotation); Q is rotated
  const float* rope_sin;     // in shared memory, map_k must already hold rotated keys
  // Dense: Sq <= Sk; query r at absolute position Sk - Sq + r. Packed: B sequences, Sq / Sk the
  // total query / key rows, maps [Hq, Sq, D] and [Hkv, Sk, D].
  int B, Hq, Hkv, Sq, Sk, D, causal;
  float scale_log2;          // scale * log2(e)
  int* status;               // device status word
  float* part;               // split forward: the parts' O tiles and (m, l) (nullptr: never split)
};

// The split plans of the forward and the backward (small problems: see FwdSplit, BwdSplit) assume
// one wave of kPlanCtas CTAs, a GB300's SM count, so that neither they nor the workspace sizes
// depend on the device.
constexpr int kPlanCtas = 152;

// Key-range split of the dense forward (fwd.cu): on small grids the key tiles of the longest
// query-tile pairs are cut into parts of at most kcap key tiles (of tile A), one CTA each, merged
// by the associative (m, l, O) combine. kcap = 0: no pair is split.
struct FwdSplit {
  int kcap;          // key tiles of tile A per part (0: no split)
  int n_pairs;       // query-tile pairs per (batch entry, head)
  int ctas_y;        // grid rows: the pairs' parts
  int parts_per_bh;  // slots one (batch entry, head) keeps: the parts of its split pairs
  int split_pairs;   // pairs cut into more than one part (merged by the combine kernel)
};

// The split for these sizes (computed once per size and cached; it does not depend on the device).
FwdSplit fwd_split_plan(int BH, int Sq, int Sk, int causal, int D);

// Workspace of the split forward: one slot per part of a split pair, holding for its tiles A and B
// the unnormalised O tile as float4 columns [D/4][128 rows] followed by m[128] and l[128];
// sized for the larger of the causal and the non-causal plan. 0: never split.
__host__ __device__ inline size_t fwd_slot_floats(int D) { return 2 * ((size_t)kTile * D + 2 * kTile); }
struct FwdWorkspace {
  size_t total;
};
FwdWorkspace fwd_workspace_layout(int B, int Hq, int Sq, int Sk, int D);

struct BwdArgs {
  const CUtensorMap* map_q;    // [B*Hq, S, D] bf16
  const CUtensorMap* map_k;    // [B*Hkv, S, D] bf16
  const CUtensorMap* map_v;
  const CUtensorMap* map_do;   // [B*Hq, S, D] bf16
  const CUtensorMap* map_dqacc;// [B*Hq, S, D] f32, box {32, 128, 1}, 128B swizzle
  const CUtensorMap* map_dq;   // [B*Hq, S, D] bf16 (deterministic path: dQ stored by TMA)
  const void* o;               // bf16 [B, Hq, S, D]
  const void* dO;              // bf16 [B, Hq, S, D]
  const float* lse;            // f32 [B, Hq, S]
  void* dq;                    // bf16 [B, Hq, S, D]
  void* dk;                    // bf16 [B, Hkv, S, D]
  void* dv;
  float* dvec;                 // f32 [B*Hq, S_pad]: D_i = rowsum(dO * O)
  float* nlse2;                // f32 [B*Hq, S_pad]: -LSE * log2(e), -inf past S
  float* dq_acc;               // f32 [B*Hq, S, D]
  float* part;                 // split key tiles' f32 dK / dV partials (dense batches; see BwdSplit)
  unsigned* tickets;           // [B*Hkv*ceil(S/128)] arrival counters of the split key tiles' parts
  const int* cu;               // packed batch: device int32 [B + 1] sequence bounds; nullptr = dense
  int max_seqlen;              // packed batch: bound on every sequence's length
  int deterministic;           // 1: dQ by the query-major kernel (dense batches only)
  const float* rope_cos;       // rotary tables f32 [S, D/2] (nullptr: none): map_q holds rotated
  const float* rope_sin;       // queries, K is rotated in shared memory, dK and dQ are turned back
  // Packed batch: B sequences, S = total rows, tensors [H, S, D], dvec / lse2 [Hq*S + kRowPad]
  // with no per-head padding.
  int B, Hq, Hkv, S, D, causal;
  float scale, scale_log2;
  int* status;
};

// Query rows (G heads x Sq new queries) one decode CTA handles for a KV head.
constexpr int kMaxDecodeRows = 16;
// Decode streams the cache in tiles of 64 keys (64-row TMA boxes), two CTAs per SM.
constexpr int kDecodeKeys = 64;
constexpr int kDecodeCtasPerSm = 2;

struct DecodeArgs {
  const CUtensorMap* map_k;  // [B*Hkv, Sk, D] bf16 cache
  const CUtensorMap* map_v;
  const void* q;             // bf16 [B, Hq, Sq, D]
  void* o;                   // bf16 [B, Hq, Sq, D]
  float* lse;                // f32 [B, Hq, Sq]
  float* part_acc;           // f32 [B*Hkv, splits, rows, D]
  float* part_ml;            // f32 [B*Hkv, splits, rows, 2]
  unsigned* tickets;         // [B*Hkv] arrival counters of the chunks, zeroed by the launcher
  int B, Hq, Hkv, Sq, Sk, D, causal, splits, chunk;
  float scale_log2;
  int* status;
};

// Workspace sections of the backward (byte offsets, each 256-aligned).
struct BwdWorkspace {
  size_t dvec_off, lse2_off, dqacc_off, part_off, ticket_off, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Split of the dense backward's key tiles. A key tile's CTA works through G * (visible query tiles)
// steps; when the problem is small, the key tiles with the most steps are cut into parts of at
// most `cap` consecutive steps, each part a CTA of its own, so that the grid fills the machine and
// no CTA is much longer than the others. Each part of a split key tile writes its f32 dK / dV
// partial to the workspace; the part that finishes last adds the parts up in part order (the
// result does not depend on the order of arrival) and writes dK, dV. cap = 0: no key tile is split.
struct BwdSplit {
  int cap;              // steps per part (0: no split)
  int ctas_per_group;   // CTAs of one (batch entry, KV head) group: sum over key tiles of their parts
  int parts_per_group;  // partials one group keeps: the parts of its split key tiles
};

inline int bwd_tile_steps(int jt, int n_tiles, int G, int causal) { return G * (causal ? n_tiles - jt : n_tiles); }

// The split the backward uses for these sizes (bwd.cu; computed once per size and cached). It does
// not depend on the device, so neither does the workspace size.
BwdSplit bwd_split_plan(int B, int Hkv, int G, int n_tiles, int causal);

inline BwdWorkspace bwd_workspace_layout(int B, int Hq, int Hkv, int S, int D) {
  BwdWorkspace w;
  const int n_tiles = ceil_div(S, kTile);
  const size_t rows_pad = (size_t)B * Hq * (size_t)n_tiles * kTile;
  w.dvec_off = 0;
  w.lse2_off = align256(w.dvec_off + rows_pad * sizeof(float));
  w.dqacc_off = align256(w.lse2_off + rows_pad * sizeof(float));
  w.part_off = align256(w.dqacc_off + (size_t)B * Hq * S * D * sizeof(float));
  // partials for the larger of the causal and the non-causal plan
  int parts = 0;
  for (int causal = 0; causal < 2; ++causal) {
    const int pp = bwd_split_plan(B, Hkv, Hq / Hkv, n_tiles, causal).parts_per_group;
    parts = pp > parts ? pp : parts;
  }
  w.ticket_off = align256(w.part_off + (size_t)B * Hkv * parts * kTile * D * 2 * sizeof(float));
  w.total = align256(w.ticket_off + (size_t)B * Hkv * n_tiles * sizeof(unsigned));
  return w;
}

// Packed batches: the D and LSE2 rows are [Hq * T] plus kRowPad rows of padding, enough for the
// widened (16-byte aligned) 132-row copies of the last query tile.
constexpr int kRowPad = 256;

inline BwdWorkspace bwd_workspace_layout_packed(int Hq, int T, int D) {
  BwdWorkspace w;
  const size_t rows = (size_t)Hq * T + kRowPad;
  w.dvec_off = 0;
  w.lse2_off = align256(w.dvec_off + rows * sizeof(float));
  w.dqacc_off = align256(w.lse2_off + rows * sizeof(float));
  w.part_off = w.ticket_off = w.total = align256(w.dqacc_off + (size_t)Hq * T * D * sizeof(float));
  return w;
}

// Tracing hooks (api.cu): no-ops unless the calling host thread armed tracing.
enum KernelKind {
  kKernelFwd = 0,
  kKernelBwdPrep = 1,
  kKernelBwdMain = 2,
  kKernelBwdConvert = 3,
  kKernelDecodeSplit = 4,
  kKernelDecodeCombine = 5,
  kKernelBwdDkdv = 6,
  kKernelBwdDq = 7,
  kKernelRope = 8,
  kKernelFwdCombine = 9,
  kKernelCount = 10
};
void trace_begin(int kind, cudaStream_t s);
void trace_end(int kind, cudaStream_t s);

// Keeps e as this host thread's last CUDA error and returns GQA_ERR_CUDA (api.cu).
int record_cuda_error(cudaError_t e);

// Once per (kernel, device): raises the kernel's dynamic shared-memory limit to smem_bytes and,
// when regs_needed > 0, checks that threads x (registers per thread at launch) covers
// regs_needed (a setmaxnreg split that the launch cannot satisfy would wait forever). Later calls
// return the cached result without calling CUDA (api.cu).
cudaError_t kernel_setup(const void* func, int smem_bytes, int threads, int regs_needed);

// Host-side size and scale checks shared by the dense entry points: GQA_OK or the error code the
// entry point returns (api.cu).
int check_common(int B, int Hq, int Hkv, int S, int D, float scale);

// Number of SMs of the current device, looked up once per device (api.cu).
int device_sm_count();

// Host launchers (fwd.cu, bwd.cu). Return a cudaError_t.
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_rope_rotate(const void* x, void* y, const float* cs, const float* sn, long long rows, int S, int D,
                               int* status, cudaStream_t stream);
cudaError_t launch_rope_convert(const float* acc, void* dq, const float* cs, const float* sn, long long rows, int S,
                                int D, float scale, int* status, cudaStream_t stream);
cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

}  // namespace gqa
