// Device-side helpers shared by the kernels of the tensor/sequence-parallel MLP
// block: inline-PTX wrappers for mbarrier, TMA and tcgen05 (sm_103a), the
// element-wise activations and the epilogue parameter block.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tpmlp.h"

namespace tpmlp {

enum DType : int { DT_F32 = TPMLP_F32, DT_F16 = TPMLP_F16, DT_BF16 = TPMLP_BF16 };
enum Act : int {
  ACT_GELU = TPMLP_ACT_GELU_TANH,
  ACT_SWIGLU = TPMLP_ACT_SWIGLU,
  ACT_IDENTITY = TPMLP_ACT_IDENTITY,
  ACT_RELU = TPMLP_ACT_RELU
};

// Device status word values (also the host-visible status codes' magnitudes).
constexpr unsigned STATUS_TIMEOUT = 6u;

// Epilogue kinds of a GEMM C[m,n] = Σ_k A(m,k)·B(n,k) accumulated in float32.
enum EpiKind : int {
  EPI_STORE = 0,  // out[m,n] = C (storage type); optional SP dim-0 scatter of rows
  EPI_F32 = 1,    // out[part][m][n] = C in float32 (one partial sum per tensor shard)
  EPI_ACT = 2,    // out = U = C, out2 = Y = act(C)        (fc1 forward)
  EPI_DACT = 3,   // out = dU = act'(aux = U) ⊙ C           (fc2 input gradient)
  EPI_ACC_F32 = 4 // out[m,n] += C in float32 (weight gradient into a float32 main_grad)
};

struct EpiParams {
  int32_t kind;
  int32_t act;
  void* out;
  int64_t ldo;
  int64_t part_stride;  // EPI_F32: elements between consecutive partials
  void* out2;
  int64_t ldo2;
  const void* aux;
  int64_t ldaux;
  int64_t swiglu_F;  // SwiGLU: column offset of the up half inside U / dU
  int32_t scatter;   // EPI_STORE: rows go to SP chunk buffers
  int32_t nshards;
  int64_t rows_per_shard;
  void* shard[TPMLP_MAX_TP];
};

// --------------------------------------------------------------------------
// Activations.  PRECISE selects libm-accurate tanhf/expf (float32 path); the
// 16-bit paths use the hardware tanh.approx.f32 and __expf, whose error is far
// below the storage rounding.
// GeLU is the tanh form of Hendrycks & Gimpel: 0.5·x·(1 + tanh(√(2/π)(x + 0.044715x³))).
// --------------------------------------------------------------------------
constexpr float kGeluC = 0.7978845608028654f;  // √(2/π)
constexpr float kGeluK = 0.044715f;

__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool PRECISE>
__device__ __forceinline__ float gelu_fwd(float x) {
  const float u = kGeluC * fmaf(kGeluK * x * x, x, x);
  const float t = PRECISE ? tanhf(u) : tanh_hw(u);
  return 0.5f * x * (1.0f + t);
}

template <bool PRECISE>
__device__ __forceinline__ float gelu_grad(float x) {
  const float u = kGeluC * fmaf(kGeluK * x * x, x, x);
  const float t = PRECISE ? tanhf(u) : tanh_hw(u);
  const float du = kGeluC * fmaf(3.0f * kGeluK, x * x, 1.0f);
  return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * du;
}

template <bool PRECISE>
__device__ __forceinline__ float sigmoid_f(float x) {
  return 1.0f / (1.0f + (PRECISE ? expf(-x) : __expf(-x)));
}

// Element-wise forward of a single-input activation (GeLU, identity, ReLU).
template <bool PRECISE>
__device__ __forceinline__ float act_fwd(int act, float x) {
  if (act == ACT_GELU) return gelu_fwd<PRECISE>(x);
  if (act == ACT_RELU) return x > 0.0f ? x : 0.0f;
  return x;
}

template <bool PRECISE>
__device__ __forceinline__ float act_grad(int act, float x) {
  if (act == ACT_GELU) return gelu_grad<PRECISE>(x);
  if (act == ACT_RELU) return x > 0.0f ? 1.0f : 0.0f;
  return 1.0f;
}

// --------------------------------------------------------------------------
// Storage conversions.
// --------------------------------------------------------------------------
template <int DT>
struct Storage;
template <>
struct Storage<DT_F32> {
  using T = float;
  static __device__ __forceinline__ float from(float x) { return x; }
  static __device__ __forceinline__ float to_f32(float x) { return x; }
};
template <>
struct Storage<DT_F16> {
  using T = __half;
  static __device__ __forceinline__ __half from(float x) { return __float2half_rn(x); }
  static __device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
};
template <>
struct Storage<DT_BF16> {
  using T = __nv_bfloat16;
  static __device__ __forceinline__ __nv_bfloat16 from(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
};

// 8 floats -> 8 16-bit values packed into a uint4 (16-byte store).
template <int DT>
__device__ __forceinline__ uint4 pack8(const float* v) {
  using S = Storage<DT>;
  uint4 r;
  typename S::T tmp[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) tmp[i] = S::from(v[i]);
  memcpy(&r, tmp, 16);
  return r;
}

template <int DT>
__device__ __forceinline__ void unpack8(const uint4& r, float* v) {
  using S = Storage<DT>;
  typename S::T tmp[8];
  memcpy(tmp, &r, 16);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = S::to_f32(tmp[i]);
}

// 128-bit read-only global load (one request per thread, no L1 allocation).
__device__ __forceinline__ uint4 ldg_nc_v4(const void* ptr) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr));
  return r;
}

__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// --------------------------------------------------------------------------
// PTX wrappers: shared-memory addresses, mbarrier, timers.
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}

// Bounded wait on phase `parity` of an mbarrier.  Gives up when *abort is set
// by another thread, or after timeout_ns (then it sets *abort and records
// STATUS_TIMEOUT in the device status word).  Returns true on completion.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, unsigned* status,
                                                  uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      if (abort_flag != nullptr) *abort_flag = 1;
      if (status != nullptr) atomicCAS(status, 0u, STATUS_TIMEOUT);
      return false;
    }
  }
}

// --------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) — 2-D tiled loads into shared memory, completing
// on an mbarrier.  c0 is the innermost (contiguous) coordinate.
// --------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// --------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory).
// --------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] · B[smem desc]ᵀ, 16-bit inputs, float32 accumulate.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on an mbarrier once all previously issued tcgen05 MMAs of this thread
// have completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Instruction descriptor of tcgen05.mma .kind::f16 (dense, no negation):
//   bits 4-5 D type (1 = f32); 7-9 A type and 10-12 B type (0 = f16, 1 = bf16);
//   bit 15 / 16 A / B major (0 = K-major, 1 = MN-major); 17-22 N >> 3; 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc_f16(bool bf16, bool a_mn, bool b_mn, int M,
                                                      int N) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((static_cast<uint32_t>(N) >> 3) << 17) | ((static_cast<uint32_t>(M) >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle:
//   bits 0-13 start address >> 4; 16-29 leading byte offset >> 4;
//   32-45 stride byte offset >> 4; bits 46-48 fixed 0b001; 61-63 swizzle (2 = 128 B).
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16) |
         (static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Tensor-memory loads: lane quarter of the warp, 32 consecutive float32 columns
// per thread (shape 32x32b).  The wait is inside the same asm statement so no
// use of the registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// --------------------------------------------------------------------------
// CTA pairs (cluster of 2) for the 2-SM tcgen05 path.
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

// shared::cta address of this CTA -> shared::cluster address of the same offset
// in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// All threads of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in the peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on an
// mbarrier that may live in the peer CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

// Tensor-memory allocation shared by the CTA pair: one warp of EACH CTA of the
// pair executes these collectively.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 2-SM MMA issued by the even CTA of the pair: A rows [0,M/2) come from its
// shared memory and rows [M/2,M) from the peer's; B columns likewise in halves;
// each CTA's tensor memory receives its M/2 rows of D.
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at the same shared offset in every CTA of `mask` once
// the issuing thread's previous 2-SM MMAs have completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"(mask)
      : "memory");
}

}  // namespace tpmlp
