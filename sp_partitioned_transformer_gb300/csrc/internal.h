// Host-side internal interface between the C ABI (api.cu) and the kernel
// launchers (copy_kernels.cu, gemm_tc.cu, gemm_simt.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "common.cuh"

namespace tpmlp {

// Sets the thread-local message returned by tpmlp_last_error(); returns `code`.
int set_error(int code, const std::string& msg);

// Per-device state (SM count, address of the device status word, timeout).
// It belongs to one CUDA context of the device: when the caller tears the
// context down (cudaDeviceReset) and a new one takes its place, the next
// current_device() call refreshes it and gives it a new `generation`, and
// every cache keyed on a device (kernel attributes, streams, symbol addresses)
// compares that number before it reuses what it holds.
struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  unsigned* status = nullptr;  // device address of the status word
  size_t max_smem_optin = 0;
  size_t smem_per_sm = 0;  // shared memory of one SM (all resident CTAs)
  unsigned long long ctx_id = 0;  // unique id of the context (cuCtxGetId)
  uint64_t generation = 0;        // > 0; process-wide, changes with the context
};
// Returns TPMLP_OK and fills `info` for the current device and its context.
int current_device(DeviceInfo** info);
uint64_t wait_timeout_ns();

// One K segment of a GEMM: A rows/cols starting at `a`, B at `b`, K extent k.
// All segments of one output partial accumulate into the same accumulator in
// the order they are listed.
struct GemmSeg {
  const void* a;
  const void* b;
  int64_t k;
  int part;
};

// C[m, n] = Σ_segments Σ_k A(m, k)·B(n, k), then an epilogue.
//   A(m, k) = a[m·lda + k] (K-major) or a[k·lda + m] (MN-major); likewise B.
// For SwiGLU fc1 (swiglu_up_row > 0) the logical N is F and the B rows of the
// up half are at swiglu_up_row + n; the accumulator tile pairs each gate column
// with its up column.
struct GemmDesc {
  int dtype = DT_BF16;
  int64_t M = 0, N = 0;
  bool a_mn = false, b_mn = false;
  int64_t lda = 0, ldb = 0;
  int64_t b_rows = 0;         // B extent along N (rows of the weight), for the TMA map
  int64_t swiglu_up_row = 0;  // > 0: SwiGLU fc1 pairing
  int nparts = 1;
  std::vector<GemmSeg> segs;
  // Optional: a K-major A split along M into equal chunks of a_chunk_rows rows
  // (sequence-parallel chunks read in place: the all-gather fused into the GEMM).
  // Tensor-core path only; the segments' `a` pointers are then ignored.
  std::vector<const void*> a_chunks;
  int64_t a_chunk_rows = 0;
  EpiParams epi{};
};

// Validates tpmlp_forward's size arguments and returns the workspace it needs.
int forward_workspace_bytes(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype, int act,
                            int mode, size_t* bytes);

int launch_gemm_tc(const GemmDesc& g, cudaStream_t st);
int launch_gemm_simt(const GemmDesc& g, cudaStream_t st);

// dim-0 movement: dst[j][0:bytes) = src[j][0:bytes) for j < n (one launch).
int launch_copy_chunks(const void* const* src, void* const* dst, int n, int64_t bytes,
                       cudaStream_t st);

// out = fixed-order float32 sum of tp partials [tp][n], rounded to dtype; if
// scatter, element e goes to out[e / chunk][e % chunk], else out[0][e].
int launch_shard_sum(const float* partials, int tp, int64_t n, int dtype, int scatter,
                     int64_t chunk, void* const* out, cudaStream_t st);

int launch_wait_selftest(unsigned* status, uint64_t timeout_ns, cudaStream_t st);

// Sequence-parallel region (sp_region.cu); x/y/dy/dx are nchunks chunk pointers
// of rpc rows each (M = nchunks·rpc rows of h).
int launch_ln_forward(const void* const* x, const void* gamma, const void* beta, float eps, void* const* y,
                      float* mean, float* rstd, int64_t M, int64_t h, int64_t rpc, int nchunks, int dtype,
                      cudaStream_t st);
int launch_ln_backward(const void* const* x, const void* gamma, const float* mean, const float* rstd,
                       const void* const* dy, void* const* dx, int accumulate, float* dgamma, float* dbeta,
                       float* part, int64_t M, int64_t h, int64_t rpc, int nchunks, int dtype, cudaStream_t st);
int launch_residual_dropout(bool forward, const void* const* r, const void* const* z, const uint8_t* const* keep,
                            float p, void* const* out, int64_t n_chunk, int nchunks, int dtype, cudaStream_t st);

// Launch accounting (tpmlp_profile_start/stop): bracket one or more kernel launches with
// CUDA events on its stream.  prof_begin returns -1 when accounting is off.
enum ProfKind : int {
  PROF_GEMM_TC = 0,
  PROF_GEMM_SIMT = 1,
  PROF_COPY = 2,
  PROF_SHARD_SUM = 3,
  PROF_SP_REGION = 4,
  PROF_ATTN = 5
};
int prof_begin(int kind, cudaStream_t st);
// `kernels` is the number of kernel launches the region enclosed.
void prof_end(int handle, double work, cudaStream_t st, int kernels = 1);

}  // namespace tpmlp
