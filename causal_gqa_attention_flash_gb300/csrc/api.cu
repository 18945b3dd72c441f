// C ABI of libgqa_attn.so: argument checks, tensor-map construction, the
// device status word and the kernel launches. The contract of every entry
// point is stated in include/gqa_attn.h.
#include <cmath>
#include <cstdio>
#include <mutex>
#include <vector>

#include "../../include/gqa_attn.h"
#include "../../include/gqa_attn_testing.h"
#include <nvtx3/nvToolsExt.h>

#include "common.h"
#include "ptx.cuh"

// Device status words, one per stream that has called into the library on a
// device (GQA_STATUS_STREAMS of them; slot 0 is shared by any further
// streams). Kernels OR STATUS_* bits into the word of the stream they were
// launched on; gqa_attn_get_error(stream) reads and clears that word only.
__device__ int g_gqa_status[GQA_STATUS_STREAMS];

namespace gqa {
namespace {

thread_local int t_last_cuda_error = 0;

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return GQA_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_base[kMaxDevices] = {};
// Streams that own a status word, per device: entry i owns word i + 1.
std::vector<void*> g_status_streams[kMaxDevices];

// Address of the status word of `stream` on the current device. The array's address is looked
// up once per device (with that device current); a stream is given the next free word on its
// first call, and streams beyond the array share word 0.
cudaError_t status_ptr(void* stream, int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_base[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_gqa_status);
    if (e != cudaSuccess) return e;
    g_status_base[dev] = static_cast<int*>(p);
  }
  std::vector<void*>& owners = g_status_streams[dev];
  size_t slot = 0;
  for (size_t i = 0; i < owners.size(); ++i)
    if (owners[i] == stream) slot = i + 1;
  if (slot == 0 && owners.size() + 1 < (size_t)GQA_STATUS_STREAMS) {
    owners.push_back(stream);
    slot = owners.size();
  }
  *out = g_status_base[dev] + slot;
  return cudaSuccess;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [nheads, S, D] tensor (D innermost) as a 3-D tiled map with box {inner, box_rows, 1}.
cudaError_t encode_3d(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int elem_bytes, int D, int S,
                      int nheads, int box_inner, CUtensorMapSwizzle swz, int box_rows = kTile) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)nheads};
  cuuint64_t strides[2] = {(cuuint64_t)D * elem_bytes, (cuuint64_t)S * D * elem_bytes};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_bf16(CUtensorMap* m, const void* ptr, int D, int S, int nheads) {
  return encode_3d(m, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, S, nheads, kChunk, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

int check_common(int B, int Hq, int Hkv, int S, int D, float scale) {
  if (B < 1 || Hq < 1 || Hkv < 1 || S < 1) return GQA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return GQA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return GQA_ERR_UNSUPPORTED;
  const long long tiles = (S + kTile - 1) / kTile;
  if (tiles > 65535) return GQA_ERR_UNSUPPORTED;
  // the padded D / LSE rows of the backward (B * Hq * tiles * 128) index with 32-bit ints
  if ((long long)B * Hq * tiles * kTile >= (1ll << 31)) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

namespace {

// ------------------------------------------------------------------ tracing

struct TraceRec {
  int kind;
  cudaEvent_t begin, end;
};
thread_local bool t_trace_armed = false;
thread_local std::vector<TraceRec> t_trace;
thread_local size_t t_trace_used = 0;
thread_local int t_trace_error = 0;

struct SetupRec {
  const void* func;
  int dev;
  cudaError_t result;
};
std::mutex g_setup_mu;
std::vector<SetupRec> g_setup;  // a few dozen kernel instances at most
int g_sm_count[kMaxDevices] = {};
int g_l2_bytes[kMaxDevices] = {};

}  // namespace

int record_cuda_error(cudaError_t e) { return fail_cuda(e); }

cudaError_t kernel_setup(const void* func, int smem_bytes, int threads, int regs_needed) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  for (const SetupRec& r : g_setup)
    if (r.func == func && r.dev == dev) return r.result;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess && regs_needed > 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, func);
    if (e == cudaSuccess && (long long)fa.numRegs * threads < regs_needed) e = cudaErrorInvalidConfiguration;
  }
  g_setup.push_back(SetupRec{func, dev, e});
  return e;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int n = __atomic_load_n(&g_sm_count[dev], __ATOMIC_RELAXED);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    __atomic_store_n(&g_sm_count[dev], n, __ATOMIC_RELAXED);
  }
  return n;
}

int device_l2_bytes() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = __atomic_load_n(&g_l2_bytes[dev], __ATOMIC_RELAXED);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess || n <= 0) return 0;
    __atomic_store_n(&g_l2_bytes[dev], n, __ATOMIC_RELAXED);
  }
  return n;
}

namespace {

const char* const kKernelRangeNames[kKernelCount] = {
    "fwd_kernel",          "bwd_prep_kernel",  "bwd_main_kernel",   "bwd_convert_kernel", "decode_split_kernel",
    "decode_combine",      "bwd_dkdv_kernel",  "bwd_dq_kernel",     "rope_rotate_kernel", "fwd_combine_kernel"};

// NVTX range over one entry point (a no-op unless a profiling tool is attached).
struct NvtxScope {
  explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
  ~NvtxScope() { nvtxRangePop(); }
  NvtxScope(const NvtxScope&) = delete;
  NvtxScope& operator=(const NvtxScope&) = delete;
};

}  // namespace

// Every launch is bracketed by an NVTX range named after its kernel and, when this host thread
// armed tracing, by two CUDA events on the launch's stream.
void trace_begin(int kind, cudaStream_t s) {
  nvtxRangePushA(kind >= 0 && kind < kKernelCount ? kKernelRangeNames[kind] : "gqa_kernel");
  if (!t_trace_armed) return;
  if (t_trace_used == t_trace.size()) {
    TraceRec r{kind, nullptr, nullptr};
    if (cudaEventCreate(&r.begin) != cudaSuccess || cudaEventCreate(&r.end) != cudaSuccess) {
      t_trace_error = 1;
      t_trace_armed = false;
      return;
    }
    t_trace.push_back(r);
  }
  t_trace[t_trace_used].kind = kind;
  if (cudaEventRecord(t_trace[t_trace_used].begin, s) != cudaSuccess) t_trace_error = 1;
}

void trace_end(int kind, cudaStream_t s) {
  nvtxRangePop();
  if (!t_trace_armed) return;
  (void)kind;
  if (cudaEventRecord(t_trace[t_trace_used].end, s) != cudaSuccess) t_trace_error = 1;
  ++t_trace_used;
}

}  // namespace gqa

using namespace gqa;

extern "C" {

}  // extern "C"

namespace {

// Dense forward, Sq <= Sk; with rotary tables (Sq = Sk) Q is rotated on load and k must
// already hold the rotated keys.
int fwd_dense(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Sk,
              int D, int causal, float scale, const float* rope_cos, const float* rope_sin, void* stream,
              void* workspace = nullptr, size_t workspace_bytes = 0) {
  if (!q || !k || !v || !o || !lse) return GQA_ERR_INVALID_ARG;
  if (Sq < 1 || Sq > Sk) return GQA_ERR_INVALID_ARG;
  int rc = check_common(B, Hq, Hkv, Sk, D, scale);
  if (rc != GQA_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return GQA_ERR_INVALID_ARG;
  CUtensorMap mq, mk, mv, mo;
  cudaError_t e;
  if ((e = encode_bf16(&mq, q, D, Sq, B * Hq)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mk, k, D, Sk, B * Hkv)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mv, v, D, Sk, B * Hkv)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mo, o, D, Sq, B * Hq)) != cudaSuccess) return fail_cuda(e);
  int* status = nullptr;
  if ((e = status_ptr(stream, &status)) != cudaSuccess) return fail_cuda(e);
  FwdArgs a;
  a.map_q = &mq;
  a.map_k = &mk;
  a.map_v = &mv;
  a.map_o = &mo;
  a.lse = lse;
  a.o = o;
  a.cu_q = nullptr;
  a.cu_k = nullptr;
  a.max_seqlen_q = 0;
  a.rope_cos = rope_cos;
  a.rope_sin = rope_sin;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.D = D;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  a.status = status;
  a.part = nullptr;
  if (workspace) {  // the split forward's slots
    const FwdWorkspace fw = fwd_workspace_layout(B, Hq, Sq, Sk, D);
    if (fw.total > 0) {
      if (workspace_bytes < fw.total) return GQA_ERR_WORKSPACE_TOO_SMALL;
      a.part = static_cast<float*>(workspace);
    }
  }
  if ((e = launch_fwd(a, static_cast<cudaStream_t>(stream))) != cudaSuccess) return fail_cuda(e);
  return GQA_OK;
}

}  // namespace

extern "C" {

int gqa_attn_fwd_cached(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Sq, int Sk, int D, int causal, float scale, void* stream) {
  NvtxScope nvtx_scope("gqa_attn_fwd_cached");
  return fwd_dense(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, nullptr, nullptr, stream);
}

int gqa_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int S,
                 int D, int causal, float scale, void* stream) {
  NvtxScope nvtx_scope("gqa_attn_fwd");
  return fwd_dense(q, k, v, o, lse, B, Hq, Hkv, S, S, D, causal, scale, nullptr, nullptr, stream);
}

size_t gqa_attn_fwd_splitkv_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D) {
  if (Sq < 1 || Sq > Sk || check_common(B, Hq, Hkv, Sk, D, 1.0f) != GQA_OK) return 0;
  return fwd_workspace_layout(B, Hq, Sq, Sk, D).total;
}

int gqa_attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                         size_t workspace_bytes, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                         void* stream) {
  NvtxScope nvtx_scope("gqa_attn_fwd_splitkv");
  if (workspace && !aligned(workspace, 256)) return GQA_ERR_INVALID_ARG;
  return fwd_dense(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, nullptr, nullptr, stream, workspace,
                   workspace_bytes);
}

size_t gqa_attn_fwd_rope_workspace_size(int B, int Hkv, int S, int D) {
  if (check_common(B, Hkv, Hkv, S, D, 1.0f) != GQA_OK) return 0;
  return align256((size_t)B * Hkv * S * D * 2);
}

int gqa_attn_fwd_rope(const void* q, const void* k, const void* v, const float* rope_cos, const float* rope_sin,
                      void* o, float* lse, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int S,
                      int D, int causal, float scale, void* stream) {
  NvtxScope nvtx_scope("gqa_attn_fwd_rope");
  if (!k || !rope_cos || !rope_sin || !workspace) return GQA_ERR_INVALID_ARG;
  int rc = check_common(B, Hq, Hkv, S, D, scale);
  if (rc != GQA_OK) return rc;
  if (!aligned(k, 16) || !aligned(rope_cos, 16) || !aligned(rope_sin, 16) || !aligned(workspace, 256))
    return GQA_ERR_INVALID_ARG;
  if (workspace_bytes < gqa_attn_fwd_rope_workspace_size(B, Hkv, S, D)) return GQA_ERR_WORKSPACE_TOO_SMALL;
  // The keys are re-read by every query tile of their group: rotate them once, here.
  int* status = nullptr;
  cudaError_t e = status_ptr(stream, &status);
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch_rope_rotate(k, workspace, rope_cos, rope_sin, (long long)B * Hkv * S, S, D, status,
                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  return fwd_dense(q, workspace, v, o, lse, B, Hq, Hkv, S, S, D, causal, scale, rope_cos, rope_sin, stream);
}

int gqa_attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                        const int* cu_seqlens_k, int nseq, int max_seqlen_q, int Hq, int Hkv, int Tq, int Tk, int D,
                        int causal, float scale, void* stream) {
  NvtxScope nvtx_scope("gqa_attn_fwd_varlen");
  if (!q || !k || !v || !o || !lse || !cu_seqlens_q || !cu_seqlens_k) return GQA_ERR_INVALID_ARG;
  if (nseq < 1 || Tq < 1 || Tk < 1 || max_seqlen_q < 1 || max_seqlen_q > Tq) return GQA_ERR_INVALID_ARG;
  int rc = check_common(1, Hq, Hkv, Tq > Tk ? Tq : Tk, D, scale);
  if (rc != GQA_OK) return rc;
  if ((long long)nseq * Hq >= (1ll << 31)) return GQA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
    return GQA_ERR_INVALID_ARG;
  CUtensorMap mq, mk, mv, mo;
  cudaError_t e;
  if ((e = encode_bf16(&mq, q, D, Tq, Hq)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mk, k, D, Tk, Hkv)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mv, v, D, Tk, Hkv)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mo, o, D, Tq, Hq)) != cudaSuccess) return fail_cuda(e);
  int* status = nullptr;
  if ((e = status_ptr(stream, &status)) != cudaSuccess) return fail_cuda(e);
  FwdArgs a;
  a.map_q = &mq;
  a.map_k = &mk;
  a.map_v = &mv;
  a.map_o = &mo;
  a.lse = lse;
  a.o = o;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.max_seqlen_q = max_seqlen_q;
  a.rope_cos = nullptr;
  a.rope_sin = nullptr;
  a.part = nullptr;  // packed batches are not split
  a.B = nseq;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = Tq;
  a.Sk = Tk;
  a.D = D;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  a.status = status;
  if ((e = launch_fwd(a, static_cast<cudaStream_t>(stream))) != cudaSuccess) return fail_cuda(e);
  return GQA_OK;
}

size_t gqa_attn_bwd_workspace_size(int B, int Hq, int Hkv, int S, int D) {
  if (check_common(B, Hq, Hkv, S, D, 1.0f) != GQA_OK) return 0;
  return bwd_workspace_layout(B, Hq, Hkv, S, D).total;
}

}  // extern "C"

namespace {

int bwd_dense(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dq,
              void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int S, int D,
              int causal, float scale, int deterministic, const float* rope_cos, const float* rope_sin,
              void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || !workspace) return GQA_ERR_INVALID_ARG;
  int rc = check_common(B, Hq, Hkv, S, D, scale);
  if (rc != GQA_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) || !aligned(workspace, 256))
    return GQA_ERR_INVALID_ARG;
  const BwdWorkspace ws = bwd_workspace_layout(B, Hq, Hkv, S, D);
  if (workspace_bytes < ws.total) return GQA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  CUtensorMap mq, mk, mv, mdo, macc, mdq;
  cudaError_t e;
  if ((e = encode_bf16(&mq, q, D, S, B * Hq)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mdq, dq, D, S, B * Hq)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mk, k, D, S, B * Hkv)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mv, v, D, S, B * Hkv)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mdo, dO, D, S, B * Hq)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_3d(&macc, wsb + ws.dqacc_off, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, S, B * Hq, 32,
                     CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return fail_cuda(e);
  int* status = nullptr;
  if ((e = status_ptr(stream, &status)) != cudaSuccess) return fail_cuda(e);
  BwdArgs a;
  a.map_q = &mq;
  a.map_k = &mk;
  a.map_v = &mv;
  a.map_do = &mdo;
  a.map_dqacc = &macc;
  a.map_dq = &mdq;
  a.deterministic = deterministic;
  a.rope_cos = rope_cos;
  a.rope_sin = rope_sin;
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dvec = reinterpret_cast<float*>(wsb + ws.dvec_off);
  a.nlse2 = reinterpret_cast<float*>(wsb + ws.lse2_off);
  a.dq_acc = reinterpret_cast<float*>(wsb + ws.dqacc_off);
  a.part = reinterpret_cast<float*>(wsb + ws.part_off);
  a.tickets = reinterpret_cast<unsigned*>(wsb + ws.ticket_off);
  a.cu = nullptr;
  a.max_seqlen = 0;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.S = S;
  a.D = D;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  a.status = status;
  if ((e = launch_bwd(a, static_cast<cudaStream_t>(stream))) != cudaSuccess) return fail_cuda(e);
  return GQA_OK;
}

}  // namespace

extern "C" {

int gqa_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int S,
                 int D, int causal, float scale, void* stream) {
  NvtxScope nvtx_scope("gqa_attn_bwd");
  return bwd_dense(q, k, v, o, dO, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, S, D, causal, scale, 0,
                   nullptr, nullptr, stream);
}

int gqa_attn_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dO,
                               const float* lse, void* dq, void* dk, void* dv, void* workspace,
                               size_t workspace_bytes, int B, int Hq, int Hkv, int S, int D, int causal, float scale,
                               void* stream) {
  NvtxScope nvtx_scope("gqa_attn_bwd_deterministic");
  return bwd_dense(q, k, v, o, dO, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, S, D, causal, scale, 1,
                   nullptr, nullptr, stream);
}

size_t gqa_attn_bwd_rope_workspace_size(int B, int Hq, int Hkv, int S, int D) {
  if (check_common(B, Hq, Hkv, S, D, 1.0f) != GQA_OK) return 0;
  return bwd_workspace_layout(B, Hq, Hkv, S, D).total + align256((size_t)B * Hq * S * D * 2);
}

int gqa_attn_bwd_rope(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                      const float* rope_cos, const float* rope_sin, void* dq, void* dk, void* dv, void* workspace,
                      size_t workspace_bytes, int B, int Hq, int Hkv, int S, int D, int causal, float scale,
                      void* stream) {
  NvtxScope nvtx_scope("gqa_attn_bwd_rope");
  if (!q || !rope_cos || !rope_sin || !workspace) return GQA_ERR_INVALID_ARG;
  int rc = check_common(B, Hq, Hkv, S, D, scale);
  if (rc != GQA_OK) return rc;
  if (!aligned(q, 16) || !aligned(rope_cos, 16) || !aligned(rope_sin, 16) || !aligned(workspace, 256))
    return GQA_ERR_INVALID_ARG;
  if (workspace_bytes < gqa_attn_bwd_rope_workspace_size(B, Hq, Hkv, S, D)) return GQA_ERR_WORKSPACE_TOO_SMALL;
  // The queries are re-read by every key tile that sees them: rotate them once, after the
  // backward's own workspace sections.
  const size_t bwd_bytes = bwd_workspace_layout(B, Hq, Hkv, S, D).total;
  void* q_rot = static_cast<uint8_t*>(workspace) + bwd_bytes;
  int* status = nullptr;
  cudaError_t e = status_ptr(stream, &status);
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch_rope_rotate(q, q_rot, rope_cos, rope_sin, (long long)B * Hq * S, S, D, status,
                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  return bwd_dense(q_rot, k, v, o, dO, lse, dq, dk, dv, workspace, bwd_bytes, B, Hq, Hkv, S, D, causal, scale, 0,
                   rope_cos, rope_sin, stream);
}

size_t gqa_attn_bwd_varlen_workspace_size(int Hq, int Hkv, int T, int D) {
  if (check_common(1, Hq, Hkv, T, D, 1.0f) != GQA_OK) return 0;
  if ((long long)Hq * T + kRowPad >= (1ll << 31)) return 0;
  return bwd_workspace_layout_packed(Hq, T, D).total;
}

int gqa_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                        void* dq, void* dk, void* dv, const int* cu_seqlens, int nseq, int max_seqlen, void* workspace,
                        size_t workspace_bytes, int Hq, int Hkv, int T, int D, int causal, float scale,
                        void* stream) {
  NvtxScope nvtx_scope("gqa_attn_bwd_varlen");
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || !cu_seqlens || !workspace)
    return GQA_ERR_INVALID_ARG;
  if (nseq < 1 || T < 1 || max_seqlen < 1 || max_seqlen > T) return GQA_ERR_INVALID_ARG;
  int rc = check_common(1, Hq, Hkv, T, D, scale);
  if (rc != GQA_OK) return rc;
  if ((long long)Hq * T + kRowPad >= (1ll << 31) || (long long)nseq * Hkv >= (1ll << 31)) return GQA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) || !aligned(cu_seqlens, 4) ||
      !aligned(workspace, 256))
    return GQA_ERR_INVALID_ARG;
  const BwdWorkspace ws = bwd_workspace_layout_packed(Hq, T, D);
  if (workspace_bytes < ws.total) return GQA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  CUtensorMap mq, mk, mv, mdo, macc;
  cudaError_t e;
  if ((e = encode_bf16(&mq, q, D, T, Hq)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mk, k, D, T, Hkv)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mv, v, D, T, Hkv)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_bf16(&mdo, dO, D, T, Hq)) != cudaSuccess) return fail_cuda(e);
  if ((e = encode_3d(&macc, wsb + ws.dqacc_off, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, T, Hq, 32,
                     CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return fail_cuda(e);
  int* status = nullptr;
  if ((e = status_ptr(stream, &status)) != cudaSuccess) return fail_cuda(e);
  BwdArgs a;
  a.map_q = &mq;
  a.map_k = &mk;
  a.map_v = &mv;
  a.map_do = &mdo;
  a.map_dqacc = &macc;
  a.map_dq = nullptr;
  a.deterministic = 0;
  a.rope_cos = nullptr;
  a.rope_sin = nullptr;
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dvec = reinterpret_cast<float*>(wsb + ws.dvec_off);
  a.nlse2 = reinterpret_cast<float*>(wsb + ws.lse2_off);
  a.dq_acc = reinterpret_cast<float*>(wsb + ws.dqacc_off);
  a.part = nullptr;  // packed batches split no key tile
  a.tickets = nullptr;
  a.cu = cu_seqlens;
  a.max_seqlen = max_seqlen;
  a.B = nseq;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.S = T;
  a.D = D;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  a.status = status;
  if ((e = launch_bwd(a, static_cast<cudaStream_t>(stream))) != cudaSuccess) return fail_cuda(e);
  return GQA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ decode

namespace gqa {
namespace {

// Key chunk per split (a multiple of the 128-key tile) and the number of non-empty splits.
// Automatic choice: the split count that minimises (waves of CTAs) x (key tiles per CTA + one
// tile's worth of per-CTA overhead), one decode CTA per SM, so that the last wave is not mostly
// empty and CTAs are not too short.
void decode_split_plan(int B, int Hkv, int Sk, int num_splits, int* splits, int* chunk) {
  const int tiles = (Sk + kDecodeKeys - 1) / kDecodeKeys;
  int s = num_splits;
  if (s <= 0) {
    const long long units = (long long)B * Hkv;
    const long long sms = (long long)device_sm_count() * kDecodeCtasPerSm;  // CTAs resident at once
    long long best = -1;
    s = 1;
    for (int c = 1; c <= tiles && c <= 512; ++c) {
      const long long per = (tiles + c - 1) / c;
      const long long waves = (units * c + sms - 1) / sms;
      const long long cost = waves * (per + 1) * 64 + c;  // small tie-break toward fewer chunks
      if (best < 0 || cost < best) {
        best = cost;
        s = c;
      }
    }
  }
  if (s > tiles) s = tiles;
  if (s < 1) s = 1;
  const int tiles_per = (tiles + s - 1) / s;
  *chunk = tiles_per * kDecodeKeys;
  *splits = (tiles + tiles_per - 1) / tiles_per;
}

int decode_rows_padded(int R) { return R <= 1 ? 1 : R <= 2 ? 2 : R <= 4 ? 4 : R <= 8 ? 8 : 16; }

int check_decode(int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || Sq > Sk || Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return GQA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return GQA_ERR_UNSUPPORTED;
  if ((Hq / Hkv) * Sq > kMaxDecodeRows) return GQA_ERR_UNSUPPORTED;
  if ((long long)B * Hkv >= 65536 || (long long)B * Hq * Sq >= (1ll << 26)) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

// Workspace: the chunks' partial accumulators, their (m, l) pairs, and one arrival ticket per
// (batch, KV head).
size_t decode_workspace(int B, int Hq, int Hkv, int Sq, int Sk, int D, int num_splits, size_t* ml_off,
                        size_t* ticket_off) {
  int splits = 1, chunk = kDecodeKeys;
  decode_split_plan(B, Hkv, Sk, num_splits, &splits, &chunk);
  const size_t rows = (size_t)B * Hkv * splits * decode_rows_padded((Hq / Hkv) * Sq);
  *ml_off = align256(rows * D * sizeof(float));
  *ticket_off = align256(*ml_off + rows * 2 * sizeof(float));
  return align256(*ticket_off + (size_t)B * Hkv * sizeof(unsigned));
}

}  // namespace
}  // namespace gqa

extern "C" {

size_t gqa_attn_decode_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D, int num_splits) {
  if (check_decode(B, Hq, Hkv, Sq, Sk, D, 1.0f) != GQA_OK) return 0;
  size_t ml = 0, tk = 0;
  return decode_workspace(B, Hq, Hkv, Sq, Sk, D, num_splits, &ml, &tk);
}

int gqa_attn_decode_fwd(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                        void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                        int causal, float scale, int num_splits, void* stream) {
  NvtxScope nvtx_scope("gqa_attn_decode_fwd");
  if (!q || !k_cache || !v_cache || !o || !lse || !workspace) return GQA_ERR_INVALID_ARG;
  int rc = check_decode(B, Hq, Hkv, Sq, Sk, D, scale);
  if (rc != GQA_OK) return rc;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(workspace, 256))
    return GQA_ERR_INVALID_ARG;
  size_t ml_off = 0, ticket_off = 0;
  const size_t need = decode_workspace(B, Hq, Hkv, Sq, Sk, D, num_splits, &ml_off, &ticket_off);
  if (workspace_bytes < need) return GQA_ERR_WORKSPACE_TOO_SMALL;
  CUtensorMap mk, mv;
  cudaError_t e;
  if ((e = encode_3d(&mk, k_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Sk, B * Hkv, kChunk,
                     CU_TENSOR_MAP_SWIZZLE_128B, kDecodeKeys)) != cudaSuccess)
    return fail_cuda(e);
  if ((e = encode_3d(&mv, v_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Sk, B * Hkv, kChunk,
                     CU_TENSOR_MAP_SWIZZLE_128B, kDecodeKeys)) != cudaSuccess)
    return fail_cuda(e);
  int* status = nullptr;
  if ((e = status_ptr(stream, &status)) != cudaSuccess) return fail_cuda(e);
  DecodeArgs a;
  a.map_k = &mk;
  a.map_v = &mv;
  a.q = q;
  a.o = o;
  a.lse = lse;
  a.part_acc = static_cast<float*>(workspace);
  a.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ml_off);
  a.tickets = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(workspace) + ticket_off);
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.D = D;
  a.causal = causal ? 1 : 0;
  decode_split_plan(B, Hkv, Sk, num_splits, &a.splits, &a.chunk);
  a.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  a.status = status;
  if ((e = launch_decode(a, static_cast<cudaStream_t>(stream))) != cudaSuccess) return fail_cuda(e);
  return GQA_OK;
}

int gqa_attn_get_error(void* stream) {
  NvtxScope nvtx_scope("gqa_attn_get_error");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  int* status = nullptr;
  if ((e = status_ptr(stream, &status)) != cudaSuccess) return fail_cuda(e);
  int h = 0;
  if ((e = cudaMemcpyAsync(&h, status, sizeof(int), cudaMemcpyDeviceToHost, s)) != cudaSuccess) return fail_cuda(e);
  if ((e = cudaMemsetAsync(status, 0, sizeof(int), s)) != cudaSuccess) return fail_cuda(e);
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail_cuda(e);
  if (h & STATUS_BOUNDS) return GQA_ERR_BOUNDS;
  if (h & STATUS_TIMEOUT) return GQA_ERR_TIMEOUT;
  if (h & STATUS_MISALIGNED_SMEM) return GQA_ERR_INTERNAL;
  if (h & STATUS_BAD_SEQLENS) return GQA_ERR_INVALID_ARG;
  return GQA_OK;
}

const char* gqa_attn_strerror(int code) {
  switch (code) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARG: return "invalid argument";
    case GQA_ERR_UNSUPPORTED: return "unsupported size (D must be 64 or 128; sizes within index range)";
    case GQA_ERR_WORKSPACE_TOO_SMALL: return "backward workspace too small";
    case GQA_ERR_CUDA: return "CUDA error";
    case GQA_ERR_TIMEOUT: return "device-side wait exceeded its time limit";
    case GQA_ERR_INTERNAL: return "kernel layout self-check failed (no work was done)";
    case GQA_ERR_BOUNDS: return "debug build: a computed coordinate fell outside its tensor (the access was skipped)";
    default: return "unknown error code";
  }
}

int gqa_attn_last_cuda_error(void) { return t_last_cuda_error; }

int gqa_attn_trace_arm(void) {
  t_trace_armed = true;
  t_trace_used = 0;
  t_trace_error = 0;
  return GQA_OK;
}

int gqa_attn_trace_collect(int* launches, double* total_ms) {
  if (!launches || !total_ms) return GQA_ERR_INVALID_ARG;
  t_trace_armed = false;
  for (int k = 0; k < kKernelCount; ++k) {
    launches[k] = 0;
    total_ms[k] = 0.0;
  }
  if (t_trace_error) return GQA_ERR_CUDA;
  for (size_t i = 0; i < t_trace_used; ++i) {
    const TraceRec& r = t_trace[i];
    cudaError_t e = cudaEventSynchronize(r.end);
    if (e != cudaSuccess) return fail_cuda(e);
    float ms = 0.f;
    if ((e = cudaEventElapsedTime(&ms, r.begin, r.end)) != cudaSuccess) return fail_cuda(e);
    launches[r.kind] += 1;
    total_ms[r.kind] += ms;
  }
  t_trace_used = 0;
  return GQA_OK;
}

int gqa_attn_selftest_wait_timeout(int limit_us, void* stream) {
  NvtxScope nvtx_scope("gqa_attn_selftest_wait_timeout");
  if (limit_us < 1 || limit_us > 1000000) return GQA_ERR_INVALID_ARG;
  int* status = nullptr;
  cudaError_t e;
  if ((e = status_ptr(stream, &status)) != cudaSuccess) return fail_cuda(e);
  if ((e = launch_wait_selftest(status, (uint64_t)limit_us * 1000ull, static_cast<cudaStream_t>(stream))) !=
      cudaSuccess)
    return fail_cuda(e);
  return GQA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ bounded-wait self-test

namespace gqa {
namespace {

// One block: thread 0 initialises an mbarrier that expects one arrival nobody
// makes, then waits on it with the ordinary bounded wait. The wait gives up
// after limit_ns, sets the TIMEOUT bit and the kernel returns.
__global__ void wait_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitGuard wg{&abort_flag, status, limit_ns};
    (void)mbar_wait(&bar, 0, wg);
  }
}

}  // namespace

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace gqa
