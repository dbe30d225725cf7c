// Sequence-parallel dim-0 movement and the fixed-order shard sum.
//
// * copy_chunks: tp independent contiguous copies in one launch.  The SP split
//   takes rows [i·s/tp, (i+1)·s/tp) of dim 0 — a contiguous slice because dim 0
//   is outermost in the [s, b, h] layout — and the all-gather concatenates the
//   chunks ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §1 `s` 在前的
//   设计：通信零转置).  Both are the same tp-chunk copy with the full tensor on
//   one side.
// * shard_sum: g's forward all-reduce / SP reduce-scatter and f's backward sum on
//   one device: R = ((P_0 + P_1) + …) + P_{tp-1} in float32, rounded once to the
//   storage type; with scatter, element e of the [M, h] result goes to sequence
//   chunk e / chunk ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §5
//   table; "Sequence Parallel 与 Context Parallel", §SP：all-gather 进、
//   reduce-scatter 出).
// Both are HBM-bound streams: 16-byte vector accesses, grid-stride loops sized
// to a few CTAs per SM, read-once data loaded with the streaming cache hint.
#include <algorithm>

#include "internal.h"

namespace tpmlp {

struct ChunkPtrs {
  const void* src[TPMLP_MAX_TP];
  void* dst[TPMLP_MAX_TP];
};

template <typename V>
__global__ void __launch_bounds__(256) copy_chunks_kernel(ChunkPtrs p, int64_t nvec) {
  const V* __restrict__ s = static_cast<const V*>(p.src[blockIdx.y]);
  V* __restrict__ d = static_cast<V*>(p.dst[blockIdx.y]);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    const V v0 = __ldcs(s + i);
    const V v1 = __ldcs(s + i + stride);
    const V v2 = __ldcs(s + i + 2 * stride);
    const V v3 = __ldcs(s + i + 3 * stride);
    d[i] = v0;
    d[i + stride] = v1;
    d[i + 2 * stride] = v2;
    d[i + 3 * stride] = v3;
  }
  for (; i < nvec; i += stride) d[i] = __ldcs(s + i);
}

// TMA bulk copy: one thread per CTA streams 32 KB slabs global -> shared ->
// global with cp.async.bulk (double-buffered, completion on an mbarrier for the
// load, bulk-group accounting for the store).  Address generation is left to
// the TMA unit; three such CTAs per SM keep enough bytes in flight.
constexpr int BULK_SLAB = 32768;

__global__ void __launch_bounds__(32) copy_chunks_bulk_kernel(ChunkPtrs p, int64_t bytes, int64_t slabs_per_chunk,
                                                              int64_t total_slabs, unsigned* status,
                                                              uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t slab[];
  __shared__ __align__(8) uint64_t bar[2];
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar[0]), 1);
  mbar_init(smem_u32(&bar[1]), 1);
  fence_barrier_init();
  uint32_t phase[2] = {0u, 0u};
  int buf = 0;
  for (int64_t t = blockIdx.x; t < total_slabs; t += gridDim.x) {
    const int64_t j = t / slabs_per_chunk;
    const int64_t off = (t - j * slabs_per_chunk) * BULK_SLAB;
    const int64_t left = bytes - off;
    const uint32_t len = static_cast<uint32_t>(left < BULK_SLAB ? left : BULK_SLAB);
    const uint32_t s = smem_u32(slab + buf * BULK_SLAB);
    const uint32_t b = smem_u32(&bar[buf]);
    // the bulk store issued from this buffer two slabs ago has finished reading it
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
    mbar_arrive_expect_tx(b, len);
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(s),
                 "l"(static_cast<const uint8_t*>(p.src[j]) + off), "r"(len), "r"(b)
                 : "memory");
    if (!mbar_wait_bounded(b, phase[buf], nullptr, status, timeout_ns)) break;
    phase[buf] ^= 1u;
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(static_cast<uint8_t*>(p.dst[j]) + off),
                 "r"(s), "r"(len)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    buf ^= 1;
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Byte copy for sizes or addresses that are not even 4-byte aligned.
__global__ void __launch_bounds__(256) copy_chunks_bytes(ChunkPtrs p, int64_t n) {
  const uint8_t* __restrict__ s = static_cast<const uint8_t*>(p.src[blockIdx.y]);
  uint8_t* __restrict__ d = static_cast<uint8_t*>(p.dst[blockIdx.y]);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    d[i] = s[i];
}

static int grid_for(int64_t units_per_chunk, int nchunks, int threads, int64_t units_per_thread) {
  DeviceInfo* dev = nullptr;
  int sms = 148;
  if (current_device(&dev) == TPMLP_OK && dev) sms = dev->num_sms;
  const int64_t want = (units_per_chunk + threads * units_per_thread - 1) / (threads * units_per_thread);
  // About 8 CTAs of 256 threads per SM in total across the tp chunks.
  const int64_t cap = std::max<int64_t>(1, (static_cast<int64_t>(sms) * 8 + nchunks - 1) / nchunks);
  return static_cast<int>(std::max<int64_t>(1, std::min(want, cap)));
}

int launch_copy_chunks(const void* const* src, void* const* dst, int n, int64_t bytes,
                       cudaStream_t st) {
  if (n <= 0 || bytes <= 0) return TPMLP_OK;
  if (n > TPMLP_MAX_TP) return set_error(TPMLP_ERR_INVALID_ARG, "too many chunks");
  ChunkPtrs p{};
  uintptr_t align_or = static_cast<uintptr_t>(bytes);
  for (int j = 0; j < n; ++j) {
    p.src[j] = src[j];
    p.dst[j] = dst[j];
    align_or |= reinterpret_cast<uintptr_t>(src[j]) | reinterpret_cast<uintptr_t>(dst[j]);
  }
  DeviceInfo* dev = nullptr;
  int rc = current_device(&dev);
  if (rc != TPMLP_OK) return rc;
  const int ph = prof_begin(PROF_COPY, st);
  if ((align_or & 15u) == 0) {
    // 16-byte aligned chunks: TMA bulk copies, 3 single-thread CTAs per SM
    static uint64_t attr_gen[64] = {};  // the device context the attribute was set in
    if (dev->device >= 0 && dev->device < 64 && attr_gen[dev->device] != dev->generation) {
      const cudaError_t e = cudaFuncSetAttribute(copy_chunks_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 2 * BULK_SLAB);
      if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
      attr_gen[dev->device] = dev->generation;
    }
    const int64_t spc = (bytes + BULK_SLAB - 1) / BULK_SLAB;
    const int64_t total = spc * n;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(total, 3 * dev->num_sms)));
    copy_chunks_bulk_kernel<<<grid, 32, 2 * BULK_SLAB, st>>>(p, bytes, spc, total, dev->status, wait_timeout_ns());
  } else if ((align_or & 3u) == 0) {
    const int64_t nvec = bytes / 4;
    dim3 grid(grid_for(nvec, n, 256, 4), n);
    copy_chunks_kernel<uint32_t><<<grid, 256, 0, st>>>(p, nvec);
  } else {
    dim3 grid(grid_for(bytes, n, 256, 4), n);
    copy_chunks_bytes<<<grid, 256, 0, st>>>(p, bytes);
  }
  prof_end(ph, 2.0 * static_cast<double>(bytes) * n, st);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("copy launch: ") + cudaGetErrorString(e));
  return TPMLP_OK;
}

// --------------------------------------------------------------------------
// Shard sum.
// --------------------------------------------------------------------------
struct OutPtrs {
  void* p[TPMLP_MAX_TP];
};

template <int DT>
__global__ void __launch_bounds__(256)
    shard_sum_vec8_kernel(const float* __restrict__ P, int tp, int64_t n, int scatter, int64_t chunk,
                          OutPtrs out) {
  using T = typename Storage<DT>::T;
  const int64_t nv = n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < nv; v += stride) {
    const int64_t e = v << 3;
    const float4 a0 = __ldcs(reinterpret_cast<const float4*>(P + e));
    const float4 a1 = __ldcs(reinterpret_cast<const float4*>(P + e + 4));
    float acc[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll 8
    for (int i = 1; i < tp; ++i) {
      const float* Pi = P + static_cast<int64_t>(i) * n + e;
      const float4 b0 = __ldcs(reinterpret_cast<const float4*>(Pi));
      const float4 b1 = __ldcs(reinterpret_cast<const float4*>(Pi + 4));
      acc[0] = __fadd_rn(acc[0], b0.x);
      acc[1] = __fadd_rn(acc[1], b0.y);
      acc[2] = __fadd_rn(acc[2], b0.z);
      acc[3] = __fadd_rn(acc[3], b0.w);
      acc[4] = __fadd_rn(acc[4], b1.x);
      acc[5] = __fadd_rn(acc[5], b1.y);
      acc[6] = __fadd_rn(acc[6], b1.z);
      acc[7] = __fadd_rn(acc[7], b1.w);
    }
    T* dst;
    if (scatter) {
      const int64_t j = e / chunk;
      dst = static_cast<T*>(out.p[j]) + (e - j * chunk);
    } else {
      dst = static_cast<T*>(out.p[0]) + e;
    }
    if constexpr (DT == DT_F32) {
      reinterpret_cast<float4*>(dst)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      *reinterpret_cast<uint4*>(dst) = pack8<DT>(acc);
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(256)
    shard_sum_scalar_kernel(const float* __restrict__ P, int tp, int64_t n, int scatter,
                            int64_t chunk, OutPtrs out) {
  using T = typename Storage<DT>::T;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += stride) {
    float acc = P[e];
    for (int i = 1; i < tp; ++i) acc = __fadd_rn(acc, P[static_cast<int64_t>(i) * n + e]);
    T* dst;
    if (scatter) {
      const int64_t j = e / chunk;
      dst = static_cast<T*>(out.p[j]) + (e - j * chunk);
    } else {
      dst = static_cast<T*>(out.p[0]) + e;
    }
    *dst = Storage<DT>::from(acc);
  }
}

template <int DT>
static void run_shard_sum(bool vec, const float* P, int tp, int64_t n, int scatter, int64_t chunk,
                          const OutPtrs& o, cudaStream_t st) {
  if (vec) {
    const int grid = grid_for(n / 8, 1, 256, 1);
    shard_sum_vec8_kernel<DT><<<grid, 256, 0, st>>>(P, tp, n, scatter, chunk, o);
  } else {
    const int grid = grid_for(n, 1, 256, 1);
    shard_sum_scalar_kernel<DT><<<grid, 256, 0, st>>>(P, tp, n, scatter, chunk, o);
  }
}

int launch_shard_sum(const float* partials, int tp, int64_t n, int dtype, int scatter, int64_t chunk,
                     void* const* out, cudaStream_t st) {
  if (n <= 0) return TPMLP_OK;
  OutPtrs o{};
  uintptr_t align_or = reinterpret_cast<uintptr_t>(partials);
  const int nout = scatter ? tp : 1;
  for (int j = 0; j < nout; ++j) {
    o.p[j] = out[j];
    align_or |= reinterpret_cast<uintptr_t>(out[j]);
  }
  const bool vec = (n % 8 == 0) && (!scatter || chunk % 8 == 0) && (align_or & 15u) == 0;
  const int ph = prof_begin(PROF_SHARD_SUM, st);
  if (dtype == DT_F32)
    run_shard_sum<DT_F32>(vec, partials, tp, n, scatter, chunk, o, st);
  else if (dtype == DT_F16)
    run_shard_sum<DT_F16>(vec, partials, tp, n, scatter, chunk, o, st);
  else
    run_shard_sum<DT_BF16>(vec, partials, tp, n, scatter, chunk, o, st);
  prof_end(ph, static_cast<double>(n) * (4.0 * tp + (dtype == DT_F32 ? 4.0 : 2.0)), st);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("shard-sum launch: ") + cudaGetErrorString(e));
  return TPMLP_OK;
}

// --------------------------------------------------------------------------
// Bounded-wait self test: one thread waits on a shared-memory mbarrier that no
// thread ever arrives at; the bounded wait must give up and record the timeout.
// --------------------------------------------------------------------------
__global__ void wait_selftest_kernel(unsigned* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile int abort_flag = 0;
    (void)mbar_wait_bounded(smem_u32(&bar), 0u, &abort_flag, status, timeout_ns);
  }
}

int launch_wait_selftest(unsigned* status, uint64_t timeout_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("selftest launch: ") + cudaGetErrorString(e));
  return TPMLP_OK;
}

}  // namespace tpmlp
