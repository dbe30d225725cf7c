// C ABI of the tensor/sequence-parallel MLP block: argument validation, the
// workspace layout and the order of launches for forward and backward.
//
// Forward ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §2 and §5 table;
// "Sequence Parallel 与 Context Parallel", §SP：all-gather 进、reduce-scatter 出):
//   [SP] all-gather X along dim 0            copy kernel      x shards -> ws.X
//   fc1 column-parallel + activation          GEMM (EPI_ACT)   U, Y
//   fc2 row-parallel + g                      PARTIALS: GEMM (EPI_F32) -> ws.P,
//                                               shard sum (all-reduce or RS) -> Z
//                                             FUSED: GEMM over all shards' K in
//                                               shard order (EPI_STORE, SP rows
//                                               scattered) -> Z
// Backward ("tensor-parallelism-matrix-split", §Backward 的通信; "Sequence Parallel
// 与 Context Parallel", §SP backward: all-gather dZ, re-gather X):
//   [SP] all-gather dZ, re-gather X           copy kernels
//   fc2 input gradient + act'                 GEMM (EPI_DACT)  dU
//   fc2 weight gradient dW2 = dZᵀ·Y           GEMM (MN-major A and B)
//   fc1 weight gradient dW1 = dUᵀ·X           GEMM (MN-major A and B)
//   fc1 input gradient + f's backward sum     as fc2 forward: partials + shard
//                                             sum, or the fused K-concatenation.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace tpmlp {

__device__ unsigned g_status_word;

static thread_local std::string g_last_error;

int set_error(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

static std::atomic<uint64_t> g_timeout_ns{2000000000ull};
uint64_t wait_timeout_ns() { return g_timeout_ns.load(); }

static std::mutex g_dev_mu;
static DeviceInfo g_devs[64];
static uint64_t g_generation = 0;

// Unique id of the calling thread's current CUDA context, 0 if it has none or
// the driver cannot say.  Ids are never reused within a process.
static unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
    ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(ptr);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

int current_device(DeviceInfo** out) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (d < 0 || d >= 64) return set_error(TPMLP_ERR_CUDA, "device ordinal out of range");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& info = g_devs[d];
  // The status word's address is looked up on every call: the lookup also makes
  // the runtime's context current on this thread, whose id then tells whether
  // the cached state still belongs to the live context.
  void* status_addr = nullptr;
  e = cudaGetSymbolAddress(&status_addr, g_status_word);
  if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
  const unsigned long long ctx = current_context_id();
  if (info.device < 0 || ctx == 0 || ctx != info.ctx_id) {
    int sms = 0, smem = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
    if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
    e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
    int smem_sm = 0;
    e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d);
    if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
    info.num_sms = sms;
    info.max_smem_optin = static_cast<size_t>(smem);
    info.smem_per_sm = static_cast<size_t>(smem_sm);
    info.device = d;
    info.ctx_id = ctx;
    info.generation = ++g_generation;
  }
  info.status = static_cast<unsigned*>(status_addr);
  *out = &info;
  return TPMLP_OK;
}

// ---------------------------------------------------------------- launch accounting
namespace {
struct ProfRec {
  int kind;
  int ev0, ev1;
  double work;
  int kernels;
};
thread_local bool g_prof_on = false;
thread_local std::vector<ProfRec> g_prof_recs;
thread_local std::vector<cudaEvent_t> g_prof_events;
thread_local uint64_t g_prof_generation = 0;  // the device context the events were made in
}  // namespace

int prof_begin(int kind, cudaStream_t st) {
  if (!g_prof_on) return -1;
  const int n = static_cast<int>(g_prof_recs.size());
  while (static_cast<int>(g_prof_events.size()) < 2 * n + 2) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return -1;
    g_prof_events.push_back(e);
  }
  if (cudaEventRecord(g_prof_events[2 * n], st) != cudaSuccess) return -1;
  g_prof_recs.push_back(ProfRec{kind, 2 * n, 2 * n + 1, 0.0, 1});
  return n;
}

void prof_end(int handle, double work, cudaStream_t st, int kernels) {
  if (handle < 0 || handle >= static_cast<int>(g_prof_recs.size())) return;
  g_prof_recs[handle].work = work;
  g_prof_recs[handle].kernels = kernels;
  cudaEventRecord(g_prof_events[g_prof_recs[handle].ev1], st);
}

// ---------------------------------------------------------------- validation
namespace {

size_t elem_size(int dt) { return dt == DT_F32 ? 4 : 2; }
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Block {
  int64_t s, b, h, f;
  int tp, sp, dtype, act, mode;
  int64_t M;   // tokens s·b
  int64_t ft;  // f / tp
  int64_t n1;  // fc1 outputs: f, or 2F for SwiGLU
  size_t e;    // storage element size
};

struct WsLayout {
  size_t x_off, dz_off, p_off, total;
};

// SP all-gather fused into the GEMMs' TMA loads: the tensor-core path reads the
// sequence chunks in place when every chunk is a whole number of 128-row blocks
// (fc1 and the fc2 input gradient pick a chunk's tensor map per row block; the
// weight gradients take each chunk as its own K segment).  Otherwise the chunks
// are first gathered into the workspace by the copy kernel.
bool fused_gather(const Block& k) {
  return k.sp && k.dtype != DT_F32 && k.tp <= 16 && ((k.s / k.tp) * k.b) % 128 == 0;
}

// forward: the forward's own layout, without the backward's gathered-dZ slot.
WsLayout ws_layout(const Block& k, bool forward = false) {
  WsLayout L{};
  size_t off = 0;
  const size_t act_bytes = static_cast<size_t>(k.M) * k.h * k.e;
  const bool gathered = k.sp && !fused_gather(k);
  L.x_off = off;
  if (gathered) off += align256(act_bytes);
  L.dz_off = off;
  if (gathered && !forward) off += align256(act_bytes);
  L.p_off = off;
  if (k.mode == TPMLP_REDUCE_PARTIALS) off += align256(static_cast<size_t>(k.tp) * k.M * k.h * 4);
  L.total = off;
  return L;
}

int check_block(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype, int act, int mode,
                Block* out) {
  if (s < 0 || b < 0) return set_error(TPMLP_ERR_INVALID_ARG, "s and b must be >= 0");
  if (h <= 0 || f <= 0) return set_error(TPMLP_ERR_INVALID_ARG, "h and f must be >= 1");
  if (tp < 1 || tp > TPMLP_MAX_TP) return set_error(TPMLP_ERR_INVALID_ARG, "tp must be in [1, 64]");
  if (sp != 0 && sp != 1) return set_error(TPMLP_ERR_INVALID_ARG, "sp must be 0 or 1");
  if (dtype < DT_F32 || dtype > DT_BF16) return set_error(TPMLP_ERR_INVALID_ARG, "unknown dtype");
  if (act < ACT_GELU || act > ACT_RELU) return set_error(TPMLP_ERR_INVALID_ARG, "unknown activation");
  if (mode != TPMLP_REDUCE_PARTIALS && mode != TPMLP_REDUCE_FUSED)
    return set_error(TPMLP_ERR_INVALID_ARG, "unknown reduce mode");
  if (s > (1ll << 31) || b > (1ll << 31) || h >= (1ll << 31) || f >= (1ll << 30))
    return set_error(TPMLP_ERR_UNSUPPORTED, "extent too large");
  const int64_t M = s * b;
  if (M >= (1ll << 31)) return set_error(TPMLP_ERR_UNSUPPORTED, "s*b >= 2^31");
  // Column/row shard widths must divide evenly (divide()/ensure_divisibility).
  if (f % tp != 0) return set_error(TPMLP_ERR_NOT_DIVISIBLE, "ffn width f is not divisible by tp");
  // SP splits dim 0 into tp equal chunks.
  if (sp && s % tp != 0)
    return set_error(TPMLP_ERR_NOT_DIVISIBLE, "First dimension of the tensor should be divisible by tensor parallel size");
  Block k{s, b, h, f, tp, sp, dtype, act, mode, M, f / tp, act == ACT_SWIGLU ? 2 * f : f, elem_size(dtype)};
  if (dtype != DT_F32) {
    if (h % 8 != 0) return set_error(TPMLP_ERR_UNSUPPORTED, "tensor-core path needs h % 8 == 0");
    if (k.ft % 8 != 0) return set_error(TPMLP_ERR_UNSUPPORTED, "tensor-core path needs (f/tp) % 8 == 0");
  }
  *out = k;
  return TPMLP_OK;
}

// Arguments of the stand-alone dim-0 operations on an [s, b, h] tensor.
int check_dim0(int64_t s, int64_t b, int64_t h, int tp, int split, int dtype, Block* out) {
  if (s < 0 || b < 0 || h < 0) return set_error(TPMLP_ERR_INVALID_ARG, "s, b and h must be >= 0");
  if (tp < 1 || tp > TPMLP_MAX_TP) return set_error(TPMLP_ERR_INVALID_ARG, "tp must be in [1, 64]");
  if (dtype < DT_F32 || dtype > DT_BF16) return set_error(TPMLP_ERR_INVALID_ARG, "unknown dtype");
  if (s > (1ll << 31) || b > (1ll << 31) || h > (1ll << 31) || s * b >= (1ll << 31))
    return set_error(TPMLP_ERR_UNSUPPORTED, "extent too large");
  if (split && s % tp != 0)
    return set_error(TPMLP_ERR_NOT_DIVISIBLE, "First dimension of the tensor should be divisible by tensor parallel size");
  *out = Block{s, b, h, tp, tp, split, dtype, ACT_IDENTITY, TPMLP_REDUCE_FUSED, s * b, 1, tp, elem_size(dtype)};
  return TPMLP_OK;
}

int check_ptr(const void* p, size_t align, const char* name) {
  if (p == nullptr) return set_error(TPMLP_ERR_INVALID_ARG, std::string(name) + " is NULL");
  if (reinterpret_cast<uintptr_t>(p) % align != 0)
    return set_error(align >= 16 ? TPMLP_ERR_UNSUPPORTED : TPMLP_ERR_INVALID_ARG,
                     std::string(name) + " is not " + std::to_string(align) + "-byte aligned");
  return TPMLP_OK;
}

int check_ptrs(const void* const* arr, int n, size_t align, const char* name) {
  if (arr == nullptr) return set_error(TPMLP_ERR_INVALID_ARG, std::string(name) + " array is NULL");
  for (int i = 0; i < n; ++i) {
    const int rc = check_ptr(arr[i], align, name);
    if (rc != TPMLP_OK) return rc;
  }
  return TPMLP_OK;
}

size_t ptr_align(const Block& k) { return k.dtype == DT_F32 ? 4 : 16; }

const uint8_t* cb(const void* p) { return static_cast<const uint8_t*>(p); }
uint8_t* wb(void* p) { return static_cast<uint8_t*>(p); }

int launch_gemm(const GemmDesc& g, cudaStream_t st) {
  return g.dtype == DT_F32 ? launch_gemm_simt(g, st) : launch_gemm_tc(g, st);
}

// The SP chunks of an [s, b, h] tensor as tp contiguous pieces of one buffer.
void chunk_ptrs(const Block& k, const void* full, const void** out) {
  const size_t chunk_bytes = static_cast<size_t>(k.s / k.tp) * k.b * k.h * k.e;
  for (int j = 0; j < k.tp; ++j) out[j] = cb(full) + j * chunk_bytes;
}

int gather(const Block& k, const void* const* shards, void* full, cudaStream_t st) {
  const void* dst_c[TPMLP_MAX_TP];
  chunk_ptrs(k, full, dst_c);
  void* dst[TPMLP_MAX_TP];
  for (int j = 0; j < k.tp; ++j) dst[j] = const_cast<void*>(dst_c[j]);
  const int64_t bytes = (k.s / k.tp) * k.b * k.h * static_cast<int64_t>(k.e);
  return launch_copy_chunks(shards, dst, k.tp, bytes, st);
}

// g / f-backward over the float32 partials in the workspace: fixed-order shard
// sum, rounded once, dim-0 chunks scattered to the SP buffers.
int shard_sum_partials(const Block& k, void* const* out, void* ws, const WsLayout& L, cudaStream_t st) {
  return launch_shard_sum(reinterpret_cast<const float*>(wb(ws) + L.p_off), k.tp, k.M * k.h, k.dtype, k.sp,
                          (k.s / k.tp) * k.b * k.h, out, st);
}

// A second stream per device, forked from and joined back into the caller's
// stream with events, so that the HBM-bound shard sum of dX runs alongside the
// tensor-bound weight-gradient GEMMs (they are independent: the weight
// gradients need no shard sum).
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  uint64_t generation = 0;  // the device context they were created in
};
std::mutex g_side_mu;
SideStream g_side[64];

int side_stream_locked(const DeviceInfo& dev, SideStream** out) {
  const int d = dev.device;
  if (d < 0 || d >= 64) return set_error(TPMLP_ERR_CUDA, "device ordinal out of range");
  SideStream& ss = g_side[d];
  if (ss.stream == nullptr || ss.generation != dev.generation) {
    // (handles of a context that was torn down are gone with it: not destroyed here)
    ss = SideStream{};
    ss.generation = dev.generation;
    cudaError_t e = cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
    if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("side stream: ") + cudaGetErrorString(e));
  }
  *out = &ss;
  return TPMLP_OK;
}

// fc2 forward (P_i = Y_i·B_i) or fc1 input gradient (G_i = dU_i·A_iᵀ) followed by g /
// f-backward: either float32 partials + shard sum, or the fused K-concatenation.
int row_parallel_and_reduce(const Block& k, bool is_dgrad, const void* a_act, const void* w,
                            void* const* out, void* ws, const WsLayout& L, cudaStream_t st,
                            bool defer_shard_sum = false) {
  const bool swiglu = k.act == ACT_SWIGLU;
  GemmDesc g;
  g.dtype = k.dtype;
  g.M = k.M;
  g.N = k.h;
  g.a_mn = false;
  if (!is_dgrad) {
    // A = Y [M, f] (K = f), B(n, k) = W2[n, k] : K-major, rows h.
    g.b_mn = false;
    g.lda = k.f;
    g.ldb = k.f;
    g.b_rows = k.h;
  } else {
    // A = dU [M, n1] (K = n1), B(n, k) = W1[k, n] : MN-major.
    g.b_mn = true;
    g.lda = k.n1;
    g.ldb = k.h;
    g.b_rows = k.n1;
  }
  // K segments: for the activation gradient of SwiGLU the shard's K range has a
  // gate part and an up part.
  auto seg = [&](int64_t kcol, int64_t klen, int part) {
    GemmSeg s;
    s.a = cb(a_act) + kcol * k.e;
    s.b = is_dgrad ? static_cast<const void*>(cb(w) + kcol * k.h * k.e) : static_cast<const void*>(cb(w) + kcol * k.e);
    s.k = klen;
    s.part = part;
    return s;
  };
  const bool two_halves = is_dgrad && swiglu;
  if (k.mode == TPMLP_REDUCE_PARTIALS) {
    g.nparts = k.tp;
    for (int i = 0; i < k.tp; ++i) {
      g.segs.push_back(seg(i * k.ft, k.ft, i));
      if (two_halves) g.segs.push_back(seg(k.f + i * k.ft, k.ft, i));
    }
    g.epi.kind = EPI_F32;
    g.epi.out = wb(ws) + L.p_off;
    g.epi.ldo = k.h;
    g.epi.part_stride = k.M * k.h;
    int rc = launch_gemm(g, st);
    if (rc != TPMLP_OK || defer_shard_sum) return rc;
    return shard_sum_partials(k, out, ws, L, st);
  }
  g.nparts = 1;
  g.segs.push_back(seg(0, k.f, 0));
  if (two_halves) g.segs.push_back(seg(k.f, k.f, 0));
  g.epi.kind = EPI_STORE;
  g.epi.ldo = k.h;
  if (k.sp) {
    g.epi.scatter = 1;
    g.epi.nshards = k.tp;
    g.epi.rows_per_shard = (k.s / k.tp) * k.b;
    for (int j = 0; j < k.tp; ++j) g.epi.shard[j] = out[j];
  } else {
    g.epi.out = out[0];
  }
  return launch_gemm(g, st);
}

}  // namespace

int forward_workspace_bytes(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype, int act,
                            int mode, size_t* bytes) {
  Block k;
  const int rc = check_block(s, b, h, f, tp, sp, dtype, act, mode, &k);
  if (rc != TPMLP_OK) return rc;
  *bytes = ws_layout(k, /*forward=*/true).total;
  return TPMLP_OK;
}

}  // namespace tpmlp

using namespace tpmlp;

// Backward pass.  main_grad: the weight gradients are added to float32
// buffers (dw1, dw2 are float*) instead of overwriting storage-type ones.
static int backward_impl(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype, int act, int mode,
                         const void* const* x, const void* w1, const void* w2, const void* u, const void* y,
                         const void* const* dz, void* const* dx, void* dw1, void* dw2, void* du, void* ws,
                         size_t ws_bytes, void* stream, bool main_grad) {
  Block k;
  int rc = check_block(s, b, h, f, tp, sp, dtype, act, mode, &k);
  if (rc != TPMLP_OK) return rc;
  const int nio = sp ? tp : 1;
  const size_t al = ptr_align(k);
  if ((rc = check_ptrs(x, nio, al, "x")) || (rc = check_ptr(w1, al, "w1")) || (rc = check_ptr(w2, al, "w2")) ||
      (rc = check_ptr(u, al, "u")) || (rc = check_ptr(y, al, "y")) || (rc = check_ptrs(dz, nio, al, "dz")) ||
      (rc = check_ptrs(dx, nio, al, "dx")) || (rc = check_ptr(dw1, main_grad ? 16 : al, "dw1")) ||
      (rc = check_ptr(dw2, main_grad ? 16 : al, "dw2")) ||
      (rc = check_ptr(du, al, "du")))
    return rc;
  const WsLayout L = ws_layout(k);
  if (L.total > 0) {
    if (ws == nullptr || ws_bytes < L.total)
      return set_error(TPMLP_ERR_WORKSPACE, "workspace needs " + std::to_string(L.total) + " bytes");
    if ((rc = check_ptr(ws, 256, "ws"))) return rc;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev))) return rc;
  if (k.M == 0) {
    // No tokens: the weight gradients are empty sums (nothing to add to main_grad).
    if (main_grad) return TPMLP_OK;
    cudaError_t e = cudaMemsetAsync(dw1, 0, static_cast<size_t>(k.n1) * h * k.e, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw2, 0, static_cast<size_t>(h) * f * k.e, st);
    if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
    return TPMLP_OK;
  }
  // [SP] g backward = all-gather of dZ; re-gather of X for the weight gradient
  // (both fused into the GEMMs' loads, or separate copies).
  const bool fused_ag = fused_gather(k);
  const int64_t rpc = sp ? (s / tp) * b : k.M;  // rows per sequence chunk
  const void* dZ = dz[0];
  const void* X = x[0];
  if (sp && !fused_ag) {
    if ((rc = gather(k, dz, wb(ws) + L.dz_off, st))) return rc;
    if ((rc = gather(k, x, wb(ws) + L.x_off, st))) return rc;
    dZ = wb(ws) + L.dz_off;
    X = wb(ws) + L.x_off;
  }
  // fc2 input gradient with the activation derivative: dU = act'(U) ⊙ (dZ·W2).
  {
    GemmDesc g;
    g.dtype = dtype;
    g.M = k.M;
    g.N = f;
    g.a_mn = false;
    g.b_mn = true;  // B(n, k) = W2[k, n]
    g.lda = h;
    g.ldb = f;
    g.b_rows = h;
    g.nparts = 1;
    g.segs.push_back(GemmSeg{dZ, w2, h, 0});
    if (fused_ag) {
      g.a_chunks.assign(dz, dz + tp);
      g.a_chunk_rows = rpc;
    }
    g.epi.kind = EPI_DACT;
    g.epi.act = act;
    g.epi.aux = u;
    g.epi.ldaux = k.n1;
    g.epi.out = du;
    g.epi.ldo = k.n1;
    g.epi.swiglu_F = act == ACT_SWIGLU ? f : 0;
    if ((rc = launch_gemm(g, st))) return rc;
  }
  auto weight_gradients = [&]() -> int {
    int rc2 = TPMLP_OK;
    // fc2 weight gradient: dW2[i, j] = Σ_m dZ[m, i]·Y[m, j]  (dB = Yᵀ·dZ stored transposed).
    {
      GemmDesc g;
      g.dtype = dtype;
      g.M = h;
      g.N = f;
      g.a_mn = true;
      g.b_mn = true;
      g.lda = h;
      g.ldb = f;
      g.b_rows = f;
      g.nparts = 1;
      if (fused_ag) {
        // K = tokens runs over the SP chunks in rank order: one K segment per chunk.
        for (int j = 0; j < tp; ++j) g.segs.push_back(GemmSeg{dz[j], cb(y) + j * rpc * f * k.e, rpc, 0});
      } else {
        g.segs.push_back(GemmSeg{dZ, y, k.M, 0});
      }
      g.epi.kind = main_grad ? EPI_ACC_F32 : EPI_STORE;
      g.epi.out = dw2;
      g.epi.ldo = f;
      if ((rc2 = launch_gemm(g, st))) return rc2;
    }
    // fc1 weight gradient: dW1[j, i] = Σ_m dU[m, j]·X[m, i]  (dA = Xᵀ·dU stored transposed).
    {
      GemmDesc g;
      g.dtype = dtype;
      g.M = k.n1;
      g.N = h;
      g.a_mn = true;
      g.b_mn = true;
      g.lda = k.n1;
      g.ldb = h;
      g.b_rows = h;
      g.nparts = 1;
      if (fused_ag) {
        for (int j = 0; j < tp; ++j) g.segs.push_back(GemmSeg{cb(du) + j * rpc * k.n1 * k.e, x[j], rpc, 0});
      } else {
        g.segs.push_back(GemmSeg{du, X, k.M, 0});
      }
      g.epi.kind = main_grad ? EPI_ACC_F32 : EPI_STORE;
      g.epi.out = dw1;
      g.epi.ldo = h;
      if ((rc2 = launch_gemm(g, st))) return rc2;
    }

    return rc2;
  };
  if (mode == TPMLP_REDUCE_PARTIALS) {
    // fc1 input-gradient partials first; their shard sum (f backward) then runs
    // on a side stream while the weight-gradient GEMMs run on the caller's.
    if ((rc = row_parallel_and_reduce(k, true, du, w1, dx, ws, L, st, /*defer_shard_sum=*/true))) return rc;
    std::lock_guard<std::mutex> lk(g_side_mu);
    SideStream* ss = nullptr;
    if ((rc = side_stream_locked(*dev, &ss))) return rc;
    cudaError_t e = cudaEventRecord(ss->fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->stream, ss->fork, 0);
    if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("fork: ") + cudaGetErrorString(e));
    rc = shard_sum_partials(k, dx, ws, L, ss->stream);
    e = cudaEventRecord(ss->join, ss->stream);
    const int rcw = weight_gradients();
    const cudaError_t e2 = cudaStreamWaitEvent(st, ss->join, 0);  // join, whatever happened above
    if (rc != TPMLP_OK) return rc;
    if (rcw != TPMLP_OK) return rcw;
    if (e != cudaSuccess || e2 != cudaSuccess)
      return set_error(TPMLP_ERR_CUDA, std::string("join: ") + cudaGetErrorString(e != cudaSuccess ? e : e2));
    return TPMLP_OK;
  }
  if ((rc = weight_gradients())) return rc;
  // fc1 input gradient + f backward (all-reduce / reduce-scatter).
  return row_parallel_and_reduce(k, true, du, w1, dx, ws, L, st);
}

extern "C" {

int tpmlp_abi_version(void) { return TPMLP_ABI_VERSION; }

const char* tpmlp_last_error(void) { return g_last_error.c_str(); }

int tpmlp_profile_start(void) {
  g_prof_recs.clear();
  DeviceInfo* dev = nullptr;
  const int rc = current_device(&dev);
  if (rc != TPMLP_OK) return rc;
  if (dev->generation != g_prof_generation) {
    g_prof_events.clear();  // events of another context: not reused, not destroyed
    g_prof_generation = dev->generation;
  }
  g_prof_on = true;
  return TPMLP_OK;
}

int tpmlp_profile_stop(tpmlp_profile* out) {
  g_prof_on = false;
  tpmlp_profile acc;
  memset(&acc, 0, sizeof(acc));
  int rc = TPMLP_OK;
  for (const ProfRec& r : g_prof_recs) {
    float ms = 0.0f;
    cudaError_t e = cudaEventSynchronize(g_prof_events[r.ev1]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, g_prof_events[r.ev0], g_prof_events[r.ev1]);
    if (e != cudaSuccess) {
      rc = set_error(TPMLP_ERR_CUDA, std::string("profile events: ") + cudaGetErrorString(e));
      continue;
    }
    acc.launches[r.kind] += r.kernels;
    acc.ms[r.kind] += ms;
    acc.work[r.kind] += r.work;
  }
  g_prof_recs.clear();
  if (out) *out = acc;
  return rc;
}

void tpmlp_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns < 1000000ull ? 1000000ull : ns); }

size_t tpmlp_workspace_size(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype, int act,
                            int mode) {
  Block k;
  if (check_block(s, b, h, f, tp, sp, dtype, act, mode, &k) != TPMLP_OK) return 0;
  return ws_layout(k).total;
}

size_t tpmlp_forward_workspace_size(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype, int act,
                                    int mode) {
  size_t bytes = 0;
  return forward_workspace_bytes(s, b, h, f, tp, sp, dtype, act, mode, &bytes) == TPMLP_OK ? bytes : 0;
}

int tpmlp_forward(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype, int act, int mode,
                  const void* const* x, const void* w1, const void* w2, void* u, void* y, void* const* z,
                  void* ws, size_t ws_bytes, void* stream) {
  Block k;
  int rc = check_block(s, b, h, f, tp, sp, dtype, act, mode, &k);
  if (rc != TPMLP_OK) return rc;
  const int nio = sp ? tp : 1;
  const size_t al = ptr_align(k);
  if ((rc = check_ptrs(x, nio, al, "x")) || (rc = check_ptr(w1, al, "w1")) || (rc = check_ptr(w2, al, "w2")) ||
      (rc = check_ptr(u, al, "u")) || (rc = check_ptr(y, al, "y")) || (rc = check_ptrs(z, nio, al, "z")))
    return rc;
  const WsLayout L = ws_layout(k, /*forward=*/true);
  if (L.total > 0) {
    if (ws == nullptr || ws_bytes < L.total)
      return set_error(TPMLP_ERR_WORKSPACE, "workspace needs " + std::to_string(L.total) + " bytes");
    if ((rc = check_ptr(ws, 256, "ws"))) return rc;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev))) return rc;
  if (k.M == 0) return TPMLP_OK;

  // [SP] f -> all-gather of the input chunks along dim 0 (fused into fc1's loads,
  // or a separate copy).
  const bool fused_ag = fused_gather(k);
  const void* X = x[0];
  if (sp && !fused_ag) {
    if ((rc = gather(k, x, wb(ws) + L.x_off, st))) return rc;
    X = wb(ws) + L.x_off;
  }
  // fc1: U = X·W1ᵀ, Y = act(U) — every tensor shard's columns in one launch.
  GemmDesc g1;
  g1.dtype = dtype;
  g1.M = k.M;
  g1.N = f;
  g1.a_mn = false;
  g1.b_mn = false;
  g1.lda = h;
  g1.ldb = h;
  g1.b_rows = k.n1;
  g1.swiglu_up_row = act == ACT_SWIGLU ? f : 0;
  g1.nparts = 1;
  g1.segs.push_back(GemmSeg{X, w1, h, 0});
  if (fused_ag) {
    g1.a_chunks.assign(x, x + tp);
    g1.a_chunk_rows = (s / tp) * b;
  }
  g1.epi.kind = EPI_ACT;
  g1.epi.act = act;
  g1.epi.out = u;
  g1.epi.ldo = k.n1;
  g1.epi.out2 = y;
  g1.epi.ldo2 = f;
  g1.epi.swiglu_F = act == ACT_SWIGLU ? f : 0;
  if ((rc = launch_gemm(g1, st))) return rc;
  // fc2 + g.
  return row_parallel_and_reduce(k, false, y, w2, z, ws, L, st);
}

int tpmlp_backward(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype, int act, int mode,
                   const void* const* x, const void* w1, const void* w2, const void* u, const void* y,
                   const void* const* dz, void* const* dx, void* dw1, void* dw2, void* du, void* ws,
                   size_t ws_bytes, void* stream) {
  return backward_impl(s, b, h, f, tp, sp, dtype, act, mode, x, w1, w2, u, y, dz, dx, dw1, dw2, du, ws, ws_bytes,
                       stream, false);
}

int tpmlp_backward_main_grad(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype, int act,
                             int mode, const void* const* x, const void* w1, const void* w2, const void* u,
                             const void* y, const void* const* dz, void* const* dx, float* main_grad_w1,
                             float* main_grad_w2, void* du, void* ws, size_t ws_bytes, void* stream) {
  return backward_impl(s, b, h, f, tp, sp, dtype, act, mode, x, w1, w2, u, y, dz, dx, main_grad_w1, main_grad_w2,
                       du, ws, ws_bytes, stream, true);
}

int tpmlp_split_dim0(const void* full, void* const* shards, int64_t s, int64_t b, int64_t h, int tp, int dtype,
                     void* stream) {
  Block k;
  int rc = check_dim0(s, b, h, tp, 1, dtype, &k);
  if (rc != TPMLP_OK) return rc;
  if ((rc = check_ptr(full, 1, "full")) || (rc = check_ptrs(shards, tp, 1, "shards"))) return rc;
  const void* src[TPMLP_MAX_TP];
  chunk_ptrs(k, full, src);
  const int64_t bytes = (s / tp) * b * h * static_cast<int64_t>(k.e);
  return launch_copy_chunks(src, shards, tp, bytes, static_cast<cudaStream_t>(stream));
}

int tpmlp_gather_dim0(const void* const* shards, void* full, int64_t s, int64_t b, int64_t h, int tp, int dtype,
                      void* stream) {
  Block k;
  int rc = check_dim0(s, b, h, tp, 1, dtype, &k);
  if (rc != TPMLP_OK) return rc;
  if ((rc = check_ptr(full, 1, "full")) || (rc = check_ptrs(shards, tp, 1, "shards"))) return rc;
  return gather(k, shards, full, static_cast<cudaStream_t>(stream));
}

int tpmlp_reduce_scatter_dim0(const float* partials, void* const* out, int64_t s, int64_t b, int64_t h, int tp,
                              int scatter, int dtype, void* stream) {
  if (scatter != 0 && scatter != 1) return set_error(TPMLP_ERR_INVALID_ARG, "scatter must be 0 or 1");
  Block k;
  int rc = check_dim0(s, b, h, tp, scatter, dtype, &k);
  if (rc != TPMLP_OK) return rc;
  if ((rc = check_ptr(partials, 4, "partials")) || (rc = check_ptrs(out, scatter ? tp : 1, k.e, "out")))
    return rc;
  return launch_shard_sum(partials, tp, s * b * h, dtype, scatter, (scatter ? s / tp : s) * b * h, out,
                          static_cast<cudaStream_t>(stream));
}

int tpmlp_device_status(void* stream, int reset) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e));
  DeviceInfo* dev = nullptr;
  int rc = current_device(&dev);
  if (rc != TPMLP_OK) return rc;
  unsigned v = 0;
  e = cudaMemcpy(&v, dev->status, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("status read: ") + cudaGetErrorString(e));
  if (reset) {
    e = cudaMemset(dev->status, 0, sizeof(unsigned));
    if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("status reset: ") + cudaGetErrorString(e));
  }
  if (v == 0) return TPMLP_OK;
  if (v == STATUS_TIMEOUT) return set_error(TPMLP_ERR_TIMEOUT, "a kernel's bounded wait expired");
  return set_error(TPMLP_ERR_CUDA, "unknown device status " + std::to_string(v));
}

int tpmlp_wait_timeout_selftest(uint64_t timeout_ns, void* stream) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull)
    return set_error(TPMLP_ERR_INVALID_ARG, "timeout_ns must be in (0, 1e10]");
  DeviceInfo* dev = nullptr;
  int rc = current_device(&dev);
  if (rc != TPMLP_OK) return rc;
  return launch_wait_selftest(dev->status, timeout_ns, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
