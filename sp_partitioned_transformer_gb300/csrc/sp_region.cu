// The sequence-parallel region around the MLP block: LayerNorm and dropout +
// residual on the [s/tp, b, h] sequence chunks ("Sequence Parallel 与 Context
// Parallel", §SP：all-gather 进、reduce-scatter 出 — LayerNorm → linear → GeLU →
// linear → dropout, with LayerNorm and dropout on sequence chunks; "tensor-
// parallel-megatron" reading, SP section: LayerNorm, dropout and the residual are
// split along the sequence).
//
// The LayerNorm's outputs are the chunks the block's fc1 reads in place (the
// all-gather fused into its loads), so no gathered copy of the activation is
// ever made.  Everything here is token-wise and HBM-bound:
//   ln_fwd_stream_kernel  persistent CTAs stream token rows through a TMA-bulk
//                         shared-memory ring (h >= 1024, 16-byte aligned rows):
//                         mean, variance (two passes over the staged row),
//                         normalise + affine, save mean/rstd;
//   ln_bwd_stream_kernel  the same ring over (x, dy[, dx]) rows:
//                         dx = rstd·(g − mean(g) − x̂·mean(g·x̂)), g = dy·γ, written
//                         or added to the residual gradient, and each CTA's dγ, dβ
//                         partial sums over its rows; ln_bwd_reduce_parts_kernel
//                         adds the partials in a fixed order (deterministic);
//   ln_fwd_kernel / ln_bwd_rows_kernel + ln_bwd_cols*_kernel
//                         one warp per token, for narrow or unaligned rows;
//   residual_dropout_*    out = r + keep·z/(1−p) and dz = keep·dout/(1−p).
#include <algorithm>

#include "internal.h"

namespace tpmlp {
namespace {

struct ChunkSet {
  const void* in[TPMLP_MAX_TP];
  const void* in2[TPMLP_MAX_TP];
  const void* mask[TPMLP_MAX_TP];
  void* out[TPMLP_MAX_TP];
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int DT>
__device__ __forceinline__ float ld1(const void* p, int64_t i) {
  return Storage<DT>::to_f32(static_cast<const typename Storage<DT>::T*>(p)[i]);
}

template <int DT>
__device__ __forceinline__ void st1(void* p, int64_t i, float v) {
  static_cast<typename Storage<DT>::T*>(p)[i] = Storage<DT>::from(v);
}

// 8 consecutive elements (16-byte aligned for 16-bit types, 32-byte for f32).
template <int DT>
__device__ __forceinline__ void ld8(const void* p, int64_t i, float* v) {
  if constexpr (DT == DT_F32) {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    unpack8<DT>(*reinterpret_cast<const uint4*>(static_cast<const typename Storage<DT>::T*>(p) + i), v);
  }
}

template <int DT>
__device__ __forceinline__ void st8(void* p, int64_t i, const float* v) {
  if constexpr (DT == DT_F32) {
    float* q = static_cast<float*>(p) + i;
    *reinterpret_cast<float4*>(q) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(q + 4) = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    *reinterpret_cast<uint4*>(static_cast<typename Storage<DT>::T*>(p) + i) = pack8<DT>(v);
  }
}

constexpr int ROWS_PER_CTA = 8;  // one warp per token row

// ------------------------------------------------------------------ LN forward
template <int DT, bool VEC>
__global__ void __launch_bounds__(256) ln_fwd_kernel(ChunkSet cs, const void* __restrict__ gamma,
                                                     const void* __restrict__ beta, float eps,
                                                     float* __restrict__ mean, float* __restrict__ rstd, int64_t M,
                                                     int64_t h, int64_t rpc) {
  const int lane = threadIdx.x & 31;
  const int64_t m = static_cast<int64_t>(blockIdx.x) * ROWS_PER_CTA + (threadIdx.x >> 5);
  if (m >= M) return;
  const int64_t j = m / rpc;
  const int64_t off = (m - j * rpc) * h;
  const void* x = cs.in[j];
  void* y = cs.out[j];
  const float inv_h = 1.0f / static_cast<float>(h);
  float s = 0.0f;
  if (VEC) {
    for (int64_t c = lane * 8; c < h; c += 256) {
      float v[8];
      ld8<DT>(x, off + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) s += v[i];
    }
  } else {
    for (int64_t c = lane; c < h; c += 32) s += ld1<DT>(x, off + c);
  }
  const float mu = warp_sum(s) * inv_h;
  float q = 0.0f;
  if (VEC) {
    for (int64_t c = lane * 8; c < h; c += 256) {
      float v[8];
      ld8<DT>(x, off + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) q += (v[i] - mu) * (v[i] - mu);
    }
  } else {
    for (int64_t c = lane; c < h; c += 32) {
      const float d = ld1<DT>(x, off + c) - mu;
      q += d * d;
    }
  }
  const float r = 1.0f / sqrtf(warp_sum(q) * inv_h + eps);
  if (VEC) {
    for (int64_t c = lane * 8; c < h; c += 256) {
      float v[8], g[8], b[8], o[8];
      ld8<DT>(x, off + c, v);
      ld8<DT>(gamma, c, g);
      ld8<DT>(beta, c, b);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = (v[i] - mu) * r * g[i] + b[i];
      st8<DT>(y, off + c, o);
    }
  } else {
    for (int64_t c = lane; c < h; c += 32)
      st1<DT>(y, off + c, (ld1<DT>(x, off + c) - mu) * r * ld1<DT>(gamma, c) + ld1<DT>(beta, c));
  }
  if (lane == 0) {
    mean[m] = mu;
    rstd[m] = r;
  }
}

// ------------------------------------------------------------------ streamed row kernels
// Persistent CTAs of 256 threads; CTA g takes the token rows g, g + G, g + 2G, ...
// (G = grid size).  Thread 0 keeps the CTA's next S rows in flight with TMA bulk
// copies (cp.async.bulk) into a ring of S shared-memory slots, one mbarrier per
// slot, so HBM reads run S rows ahead of the arithmetic and nothing of a row is
// held in registers.  γ (and β) are staged in shared memory once per CTA.  Each
// thread owns the 8-element vectors vi = threadIdx.x + 256·k, k < V, of every row
// (h <= 256·8·V).  A slot holds `nin` rows of the token (x; or x and dy; or x, dy
// and the dx being accumulated into), each padded to 128 bytes.
constexpr int STREAM_THREADS = 256;
constexpr int STREAM_MAX_SLOTS = 8;
constexpr int STREAM_MIN_H = 1024;  // below this a warp per row is the better shape
constexpr int STREAM_MAX_V = 4;     // h <= 8192

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// 8 elements (vector vi) of a row in shared memory.
template <int DT>
__device__ __forceinline__ void lds8(const uint8_t* row, int vi, float* v) {
  if constexpr (DT == DT_F32) {
    const float4 a = reinterpret_cast<const float4*>(row)[2 * vi];
    const float4 b = reinterpret_cast<const float4*>(row)[2 * vi + 1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    unpack8<DT>(reinterpret_cast<const uint4*>(row)[vi], v);
  }
}

// Copies vector vi (8 elements) of a global array into a shared-memory row.
template <int DT>
__device__ __forceinline__ void stage8(uint8_t* row, const void* src, int vi) {
  const uint4* s = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(src) + static_cast<int64_t>(vi) * 8 *
                                                                                        sizeof(typename Storage<DT>::T));
  uint4* d = reinterpret_cast<uint4*>(row + static_cast<int64_t>(vi) * 8 * sizeof(typename Storage<DT>::T));
  d[0] = s[0];
  if constexpr (DT == DT_F32) d[1] = s[1];
}

// Sum of (a, b) over the CTA; the fixed shuffle/warp order makes it
// deterministic.  red[] must be free (a __syncthreads since its last read):
// one barrier.
__device__ __forceinline__ float2 block_sum2_free(float a, float b, float2* red) {
  a = warp_sum(a);
  b = warp_sum(b);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[w] = make_float2(a, b);
  __syncthreads();
  const float2 t = lane < STREAM_THREADS / 32 ? red[lane] : make_float2(0.0f, 0.0f);
  return make_float2(warp_sum(t.x), warp_sum(t.y));
}

struct RowRing {
  uint8_t* base;   // slot 0
  uint32_t rb;     // bytes of one row
  uint32_t rb_al;  // ... padded to 128
  int nin;         // rows per slot
  int S;           // slots
};

// Thread 0: start the bulk copies of the CTA's k-th row into slot k % S.
__device__ __forceinline__ void ring_issue(const RowRing& ring, uint64_t* full, const ChunkSet& cs, int64_t k,
                                          int64_t h, int64_t rpc, size_t esz) {
  const int64_t m = blockIdx.x + k * gridDim.x;
  const int64_t j = m / rpc;
  const int64_t off = (m - j * rpc) * h * static_cast<int64_t>(esz);
  const int s = static_cast<int>(k % ring.S);
  const uint32_t bar = smem_u32(&full[s]);
  const uint32_t dst = smem_u32(ring.base + static_cast<size_t>(s) * ring.nin * ring.rb_al);
  mbar_arrive_expect_tx(bar, ring.rb * ring.nin);
  bulk_g2s(dst, static_cast<const uint8_t*>(cs.in[j]) + off, ring.rb, bar);
  if (ring.nin > 1) bulk_g2s(dst + ring.rb_al, static_cast<const uint8_t*>(cs.in2[j]) + off, ring.rb, bar);
  if (ring.nin > 2) bulk_g2s(dst + 2 * ring.rb_al, static_cast<const uint8_t*>(cs.out[j]) + off, ring.rb, bar);
}

// Thread 0, after a timed-out wait on row k: wait (bounded) for the copies still
// in flight into this CTA's shared memory before the CTA exits.
__device__ __forceinline__ void ring_drain(const RowRing& ring, uint64_t* full, int64_t k, int64_t cnt,
                                           unsigned* status, uint64_t timeout_ns) {
  const int64_t issued = min(cnt, static_cast<int64_t>(ring.S) + (k > 0 ? k - 1 : 0));
  for (int64_t r = k; r < issued; ++r)
    if (!mbar_wait_bounded(smem_u32(&full[r % ring.S]), static_cast<uint32_t>((r / ring.S) & 1), nullptr, status,
                           timeout_ns))
      break;
}

__host__ __device__ __forceinline__ uint32_t pad128(uint32_t x) { return (x + 127u) & ~127u; }

// Shared memory: [γ | β | ring of S slots of one x row].
template <int DT, int V>
__global__ void __launch_bounds__(STREAM_THREADS) ln_fwd_stream_kernel(ChunkSet cs, const void* __restrict__ gamma,
                                                                       const void* __restrict__ beta, float eps,
                                                                       float* __restrict__ mean,
                                                                       float* __restrict__ rstd, int64_t M, int64_t h,
                                                                       int64_t rpc, int S, unsigned* status,
                                                                       uint64_t timeout_ns) {
  using T = typename Storage<DT>::T;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[STREAM_MAX_SLOTS];
  __shared__ float2 red[STREAM_THREADS / 32];
  __shared__ int abort_flag;
  const int tid = threadIdx.x;
  const int nv = static_cast<int>(h / 8);
  const uint32_t rb = static_cast<uint32_t>(h * sizeof(T));
  uint8_t* sg = smem;
  uint8_t* sb = smem + pad128(rb);
  const RowRing ring{smem + 2 * pad128(rb), rb, pad128(rb), 1, S};
  const int64_t G = gridDim.x;
  const int64_t cnt = (M - blockIdx.x + G - 1) / G;
  // each thread stages, and later reads, only its own vectors of γ and β
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int vi = tid + k * STREAM_THREADS;
    if (vi < nv) {
      stage8<DT>(sg, gamma, vi);
      stage8<DT>(sb, beta, vi);
    }
  }
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_barrier_init();
    for (int64_t k = 0; k < S && k < cnt; ++k) ring_issue(ring, full, cs, k, h, rpc, sizeof(T));
  }
  const float inv_h = 1.0f / static_cast<float>(h);
  for (int64_t k = 0; k < cnt; ++k) {
    const int s = static_cast<int>(k % S);
    if (tid == 0 &&
        !mbar_wait_bounded(smem_u32(&full[s]), static_cast<uint32_t>((k / S) & 1), nullptr, status, timeout_ns))
      abort_flag = 1;
    __syncthreads();  // row k is in slot s; every thread is done with row k - 1
    if (abort_flag) {
      if (tid == 0) ring_drain(ring, full, k, cnt, status, timeout_ns);
      return;
    }
    if (tid == 0 && k >= 1 && k - 1 + S < cnt) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ring_issue(ring, full, cs, k - 1 + S, h, rpc, sizeof(T));
    }
    const uint8_t* row = ring.base + static_cast<size_t>(s) * ring.rb_al;
    // Mean and variance from one block reduction of the shifted sums
    // Σ(x − c) and Σ(x − c)², c = the row's first element (the shifted-data
    // method: with c inside the data's range the subtraction
    // E[(x−c)²] − E[x−c]² does not cancel away the variance the way raw
    // Σx² − (Σx)²/h does when the mean is large against the spread).  red[] is
    // free: every thread passed this row's first barrier after reading it.
    const float c = Storage<DT>::to_f32(reinterpret_cast<const T*>(row)[0]);
    float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int kk = 0; kk < V; ++kk) {
      const int vi = tid + kk * STREAM_THREADS;
      if (vi < nv) {
        float v[8];
        lds8<DT>(row, vi, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float d = v[i] - c;
          s1 += d;
          s2 = fmaf(d, d, s2);
        }
      }
    }
    const float2 st = block_sum2_free(s1, s2, red);
    const float dm = st.x * inv_h;
    const float mu = c + dm;
    const float r = 1.0f / sqrtf(fmaxf(st.y * inv_h - dm * dm, 0.0f) + eps);
    const int64_t m = blockIdx.x + k * G;
    const int64_t j = m / rpc;
    T* y = static_cast<T*>(cs.out[j]) + (m - j * rpc) * h;
#pragma unroll
    for (int kk = 0; kk < V; ++kk) {
      const int vi = tid + kk * STREAM_THREADS;
      if (vi < nv) {
        float v[8], g[8], b[8], o[8];
        lds8<DT>(row, vi, v);
        lds8<DT>(sg, vi, g);
        lds8<DT>(sb, vi, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = (v[i] - mu) * r * g[i] + b[i];
        st8<DT>(y, static_cast<int64_t>(vi) * 8, o);
      }
    }
    if (tid == 0) {
      mean[m] = mu;
      rstd[m] = r;
    }
  }
}

// dx = rstd·(g − mean(g) − x̂·mean(g·x̂)), g = dy·γ, written or added to dx; and
// this CTA's partial sums of dγ = Σ dy·x̂ and dβ = Σ dy over its rows, in row
// order, stored as part[blockIdx.x][:] and part[G + blockIdx.x][:].
// Shared memory: [γ | ring of S slots of (x, dy[, dx]) rows].
template <int DT, int V>
__global__ void __launch_bounds__(STREAM_THREADS) ln_bwd_stream_kernel(ChunkSet cs, const void* __restrict__ gamma,
                                                                       const float* __restrict__ mean,
                                                                       const float* __restrict__ rstd, int accumulate,
                                                                       float* __restrict__ part, int64_t M, int64_t h,
                                                                       int64_t rpc, int S, unsigned* status,
                                                                       uint64_t timeout_ns) {
  using T = typename Storage<DT>::T;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[STREAM_MAX_SLOTS];
  __shared__ float2 red[STREAM_THREADS / 32];
  __shared__ int abort_flag;
  const int tid = threadIdx.x;
  const int nv = static_cast<int>(h / 8);
  const uint32_t rb = static_cast<uint32_t>(h * sizeof(T));
  uint8_t* sg = smem;
  const RowRing ring{smem + pad128(rb), rb, pad128(rb), accumulate ? 3 : 2, S};
  const int64_t G = gridDim.x;
  const int64_t cnt = (M - blockIdx.x + G - 1) / G;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int vi = tid + k * STREAM_THREADS;
    if (vi < nv) stage8<DT>(sg, gamma, vi);
  }
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_barrier_init();
    for (int64_t k = 0; k < S && k < cnt; ++k) ring_issue(ring, full, cs, k, h, rpc, sizeof(T));
  }
  float ag[V][8], ab[V][8];
#pragma unroll
  for (int kk = 0; kk < V; ++kk)
#pragma unroll
    for (int i = 0; i < 8; ++i) ag[kk][i] = ab[kk][i] = 0.0f;
  const float inv_h = 1.0f / static_cast<float>(h);
  float mu_next = cnt > 0 ? mean[blockIdx.x] : 0.0f;
  float r_next = cnt > 0 ? rstd[blockIdx.x] : 0.0f;
  for (int64_t k = 0; k < cnt; ++k) {
    const int s = static_cast<int>(k % S);
    const int64_t m = blockIdx.x + k * G;
    const float mu = mu_next, r = r_next;
    if (k + 1 < cnt) {  // the next row's statistics, one row ahead
      mu_next = mean[m + G];
      r_next = rstd[m + G];
    }
    if (tid == 0 &&
        !mbar_wait_bounded(smem_u32(&full[s]), static_cast<uint32_t>((k / S) & 1), nullptr, status, timeout_ns))
      abort_flag = 1;
    __syncthreads();  // row k is in slot s; every thread is done with row k - 1
    if (abort_flag) {
      if (tid == 0) ring_drain(ring, full, k, cnt, status, timeout_ns);
      return;
    }
    if (tid == 0 && k >= 1 && k - 1 + S < cnt) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ring_issue(ring, full, cs, k - 1 + S, h, rpc, sizeof(T));
    }
    const uint8_t* xs = ring.base + static_cast<size_t>(s) * ring.nin * ring.rb_al;
    const uint8_t* ds = xs + ring.rb_al;
    const uint8_t* os = xs + 2 * ring.rb_al;
    float sg1 = 0.0f, sgx = 0.0f;
#pragma unroll
    for (int kk = 0; kk < V; ++kk) {
      const int vi = tid + kk * STREAM_THREADS;
      if (vi < nv) {
        float xv[8], d[8], g[8];
        lds8<DT>(xs, vi, xv);
        lds8<DT>(ds, vi, d);
        lds8<DT>(sg, vi, g);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float xh = (xv[i] - mu) * r;
          const float gi = d[i] * g[i];
          sg1 += gi;
          sgx += gi * xh;
          ag[kk][i] += d[i] * xh;
          ab[kk][i] += d[i];
        }
      }
    }
    const float2 tot = block_sum2_free(sg1, sgx, red);  // red[] free: the row's first barrier follows its last read
    const float mg = tot.x * inv_h, mgx = tot.y * inv_h;
    const int64_t j = m / rpc;
    T* dx = static_cast<T*>(cs.out[j]) + (m - j * rpc) * h;
#pragma unroll
    for (int kk = 0; kk < V; ++kk) {
      const int vi = tid + kk * STREAM_THREADS;
      if (vi < nv) {
        float xv[8], d[8], g[8], o[8];
        lds8<DT>(xs, vi, xv);
        lds8<DT>(ds, vi, d);
        lds8<DT>(sg, vi, g);
        if (accumulate) lds8<DT>(os, vi, o);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float t = r * (d[i] * g[i] - mg - (xv[i] - mu) * r * mgx);
          o[i] = accumulate ? o[i] + t : t;
        }
        st8<DT>(dx, static_cast<int64_t>(vi) * 8, o);
      }
    }
  }
  float* pg = part + static_cast<int64_t>(blockIdx.x) * h;
  float* pb = part + (G + blockIdx.x) * h;
#pragma unroll
  for (int kk = 0; kk < V; ++kk) {
    const int vi = tid + kk * STREAM_THREADS;
    if (vi < nv) {
      float4* qg = reinterpret_cast<float4*>(pg + static_cast<int64_t>(vi) * 8);
      float4* qb = reinterpret_cast<float4*>(pb + static_cast<int64_t>(vi) * 8);
      qg[0] = make_float4(ag[kk][0], ag[kk][1], ag[kk][2], ag[kk][3]);
      qg[1] = make_float4(ag[kk][4], ag[kk][5], ag[kk][6], ag[kk][7]);
      qb[0] = make_float4(ab[kk][0], ab[kk][1], ab[kk][2], ab[kk][3]);
      qb[1] = make_float4(ab[kk][4], ab[kk][5], ab[kk][6], ab[kk][7]);
    }
  }
}

// dγ[c], dβ[c] from the G per-CTA partials (part = [dγ rows G | dβ rows G] of h):
// eight row-strided partial sums per column, then added in index order — the
// same association on every run.
__global__ void __launch_bounds__(256) ln_bwd_reduce_parts_kernel(const float* __restrict__ part,
                                                                  float* __restrict__ dgamma,
                                                                  float* __restrict__ dbeta, int64_t h, int64_t G) {
  __shared__ float acc[8][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * 32 + tx;  // over [dγ | dβ], 2h columns
  float a = 0.0f;
  if (col < 2 * h) {
    const int64_t which = col >= h ? 1 : 0;
    const float* p = part + which * G * h + (col - which * h);
#pragma unroll 4
    for (int64_t g = ty; g < G; g += 8) a += p[g * h];
  }
  acc[ty][tx] = a;
  __syncthreads();
  if (ty == 0 && col < 2 * h) {
    float t = acc[0][tx];
#pragma unroll
    for (int y = 1; y < 8; ++y) t += acc[y][tx];
    if (col < h) dgamma[col] = t;
    else dbeta[col - h] = t;
  }
}

constexpr int VCOL_ROWS = 16;  // tokens per dγ/dβ partial in the vectorised column kernel

// Eight consecutive columns per thread, VCOL_ROWS tokens per CTA row block; the
// block's chunk is computed once when chunks are whole numbers of blocks.
template <int DT>
__global__ void __launch_bounds__(256) ln_bwd_cols_vec_kernel(ChunkSet cs, const float* __restrict__ mean,
                                                              const float* __restrict__ rstd, float* __restrict__ part,
                                                              int64_t M, int64_t h, int64_t rpc, int64_t nrb) {
  const int64_t c = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
  const int64_t rb = blockIdx.y;
  if (c >= h) return;
  const int64_t m0 = rb * VCOL_ROWS, m1 = min(M, m0 + VCOL_ROWS);
  const bool one_chunk = (rpc % VCOL_ROWS) == 0;
  const int64_t j0 = m0 / rpc;
  float ag[8], ab[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) ag[i] = ab[i] = 0.0f;
#pragma unroll 4
  for (int64_t m = m0; m < m1; ++m) {
    const int64_t jj = one_chunk ? j0 : m / rpc;
    const int64_t idx = (m - jj * rpc) * h + c;
    float d[8], xv[8];
    ld8<DT>(cs.in2[jj], idx, d);
    ld8<DT>(cs.in[jj], idx, xv);
    const float mu = mean[m], r = rstd[m];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ag[i] += d[i] * (xv[i] - mu) * r;
      ab[i] += d[i];
    }
  }
  float* pg = part + rb * h + c;
  float* pb = part + (nrb + rb) * h + c;
  *reinterpret_cast<float4*>(pg) = make_float4(ag[0], ag[1], ag[2], ag[3]);
  *reinterpret_cast<float4*>(pg + 4) = make_float4(ag[4], ag[5], ag[6], ag[7]);
  *reinterpret_cast<float4*>(pb) = make_float4(ab[0], ab[1], ab[2], ab[3]);
  *reinterpret_cast<float4*>(pb + 4) = make_float4(ab[4], ab[5], ab[6], ab[7]);
}

// ------------------------------------------------------------------ LN backward
// cs.in = x chunks, cs.in2 = dy chunks, cs.out = dx chunks.
template <int DT, bool VEC>
__global__ void __launch_bounds__(256) ln_bwd_rows_kernel(ChunkSet cs, const void* __restrict__ gamma,
                                                          const float* __restrict__ mean,
                                                          const float* __restrict__ rstd, int accumulate, int64_t M,
                                                          int64_t h, int64_t rpc) {
  const int lane = threadIdx.x & 31;
  const int64_t m = static_cast<int64_t>(blockIdx.x) * ROWS_PER_CTA + (threadIdx.x >> 5);
  if (m >= M) return;
  const int64_t j = m / rpc;
  const int64_t off = (m - j * rpc) * h;
  const void* x = cs.in[j];
  const void* dy = cs.in2[j];
  void* dx = cs.out[j];
  const float mu = mean[m], r = rstd[m];
  const float inv_h = 1.0f / static_cast<float>(h);
  float sg = 0.0f, sgx = 0.0f;
  if (VEC) {
    for (int64_t c = lane * 8; c < h; c += 256) {
      float v[8], d[8], g[8];
      ld8<DT>(x, off + c, v);
      ld8<DT>(dy, off + c, d);
      ld8<DT>(gamma, c, g);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float gi = d[i] * g[i];
        sg += gi;
        sgx += gi * (v[i] - mu) * r;
      }
    }
  } else {
    for (int64_t c = lane; c < h; c += 32) {
      const float gi = ld1<DT>(dy, off + c) * ld1<DT>(gamma, c);
      sg += gi;
      sgx += gi * (ld1<DT>(x, off + c) - mu) * r;
    }
  }
  const float mg = warp_sum(sg) * inv_h, mgx = warp_sum(sgx) * inv_h;
  if (VEC) {
    for (int64_t c = lane * 8; c < h; c += 256) {
      float v[8], d[8], g[8], o[8];
      ld8<DT>(x, off + c, v);
      ld8<DT>(dy, off + c, d);
      ld8<DT>(gamma, c, g);
      if (accumulate) ld8<DT>(dx, off + c, o);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float t = r * (d[i] * g[i] - mg - (v[i] - mu) * r * mgx);
        o[i] = accumulate ? o[i] + t : t;
      }
      st8<DT>(dx, off + c, o);
    }
  } else {
    for (int64_t c = lane; c < h; c += 32) {
      const float t = r * (ld1<DT>(dy, off + c) * ld1<DT>(gamma, c) - mg - (ld1<DT>(x, off + c) - mu) * r * mgx);
      st1<DT>(dx, off + c, accumulate ? ld1<DT>(dx, off + c) + t : t);
    }
  }
}

constexpr int COL_ROWS = 128;  // tokens per dγ/dβ partial

// part[rb][c] = Σ_{m in block rb} dy·x̂ (dγ) and part[nrb + rb][c] = Σ dy (dβ).
template <int DT>
__global__ void __launch_bounds__(256) ln_bwd_cols_kernel(ChunkSet cs, const float* __restrict__ mean,
                                                          const float* __restrict__ rstd, float* __restrict__ part,
                                                          int64_t M, int64_t h, int64_t rpc, int64_t nrb) {
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t rb = blockIdx.y;
  if (c >= h) return;
  const int64_t m0 = rb * COL_ROWS, m1 = min(M, m0 + COL_ROWS);
  float ag = 0.0f, ab = 0.0f;
  for (int64_t m = m0; m < m1; ++m) {
    const int64_t j = m / rpc;
    const int64_t idx = (m - j * rpc) * h + c;
    const float d = ld1<DT>(cs.in2[j], idx);
    ag += d * (ld1<DT>(cs.in[j], idx) - mean[m]) * rstd[m];
    ab += d;
  }
  part[rb * h + c] = ag;
  part[(nrb + rb) * h + c] = ab;
}

__global__ void __launch_bounds__(256) ln_bwd_reduce_kernel(const float* __restrict__ part, float* __restrict__ dgamma,
                                                            float* __restrict__ dbeta, int64_t h, int64_t nrb) {
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= h) return;
  float ag = 0.0f, ab = 0.0f;
  for (int64_t rb = 0; rb < nrb; ++rb) {  // fixed order: deterministic
    ag += part[rb * h + c];
    ab += part[(nrb + rb) * h + c];
  }
  dgamma[c] = ag;
  dbeta[c] = ab;
}

// ------------------------------------------------------------------ dropout + residual
// forward: cs.in = r, cs.in2 = z, cs.mask = keep, cs.out = out
// backward: cs.in2 = dout, cs.mask = keep, cs.out = dz (cs.in unused)
template <int DT, bool FWD>
__global__ void __launch_bounds__(256) residual_dropout_kernel(ChunkSet cs, float scale, int64_t n_chunk) {
  const int j = blockIdx.y;
  const uint8_t* keep = static_cast<const uint8_t*>(cs.mask[j]);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_chunk; e += stride) {
    const float z = ld1<DT>(cs.in2[j], e);
    const float kz = keep[e] ? z * scale : 0.0f;
    st1<DT>(cs.out[j], e, FWD ? ld1<DT>(cs.in[j], e) + kz : kz);
  }
}

// 8 consecutive elements kept in their storage type until used (4 registers for
// 16-bit types), so that several vectors per thread can be in flight.
template <int DT>
struct Raw8 {
  uint4 w[DT == DT_F32 ? 2 : 1];
  __device__ __forceinline__ void load(const void* p, int64_t i) {
    const uint4* q = reinterpret_cast<const uint4*>(static_cast<const typename Storage<DT>::T*>(p) + i);
    w[0] = q[0];
    if constexpr (DT == DT_F32) w[1] = q[1];
  }
  __device__ __forceinline__ void unpack(float* v) const {
    if constexpr (DT == DT_F32) {
      memcpy(v, &w[0], 16);
      memcpy(v + 4, &w[1], 16);
    } else {
      unpack8<DT>(w[0], v);
    }
  }
};

template <int DT, bool FWD>
__global__ void __launch_bounds__(256) residual_dropout_vec8_kernel(ChunkSet cs, float scale, int64_t n_chunk) {
  constexpr int U = 4;  // vectors of 8 elements in flight per thread
  const int j = blockIdx.y;
  const uint8_t* keep = static_cast<const uint8_t*>(cs.mask[j]);
  const int64_t nvec = n_chunk / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t v0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v0 < nvec; v0 += U * stride) {
    Raw8<DT> z[U], r[U];
    uint2 k8[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nvec) {
        z[u].load(cs.in2[j], v * 8);
        if (FWD) r[u].load(cs.in[j], v * 8);
        k8[u] = *reinterpret_cast<const uint2*>(keep + v * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nvec) {
        const uint8_t* kb = reinterpret_cast<const uint8_t*>(&k8[u]);
        float zf[8], rf[8], o[8];
        z[u].unpack(zf);
        if (FWD) r[u].unpack(rf);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float kz = kb[i] ? zf[i] * scale : 0.0f;
          o[i] = FWD ? rf[i] + kz : kz;
        }
        st8<DT>(cs.out[j], v * 8, o);
      }
    }
  }
}

int check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return TPMLP_OK;
}

uintptr_t align_bits(const void* const* arr, int n) {
  uintptr_t a = 0;
  for (int i = 0; i < n; ++i) a |= reinterpret_cast<uintptr_t>(arr[i]);
  return a;
}

// Ring slots and grid of a streamed kernel: `fixed` bytes of staged parameters,
// then S slots of `slot` bytes, S in [2, 8] and as large as a share of the SM's
// shared memory for `ctas_per_sm` resident CTAs allows; one wave of persistent
// CTAs, at most `max_grid`.  ok = false when two slots do not fit.
struct StreamPlan {
  bool ok = false;
  int S = 0;
  int grid = 0;
  size_t smem = 0;
};

StreamPlan plan_stream(const void* fn, size_t fixed, size_t slot, int ctas_per_sm, int64_t max_grid) {
  StreamPlan p;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != TPMLP_OK || dev == nullptr || max_grid < 1) return p;
  const size_t cap = dev->max_smem_optin > 1024 ? dev->max_smem_optin - 1024 : 0;  // static shared memory
  const size_t share = dev->smem_per_sm / static_cast<size_t>(ctas_per_sm);
  const size_t budget = std::min(cap, share > 2048 ? share - 2048 : 0);
  int S = budget > fixed ? static_cast<int>(std::min<size_t>(STREAM_MAX_SLOTS, (budget - fixed) / slot)) : 0;
  S = std::max(S, 2);
  const size_t smem = fixed + static_cast<size_t>(S) * slot;
  if (smem > cap) return p;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return p;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, STREAM_THREADS, smem) != cudaSuccess || occ < 1) {
    cudaGetLastError();
    return p;
  }
  p.ok = true;
  p.S = S;
  p.smem = smem;
  p.grid = static_cast<int>(std::min<int64_t>(max_grid, static_cast<int64_t>(occ) * dev->num_sms));
  return p;
}

// Grid of a grid-stride elementwise kernel over nchunks chunks: one resident
// wave (CTAs per SM from the kernel's occupancy), at most one CTA per 256 units
// of a chunk, split evenly over the chunks (grid.y).
dim3 dropout_grid(const void* fn, int64_t units_per_chunk, int nchunks) {
  DeviceInfo* dev = nullptr;
  int sms = 148, occ = 4;
  if (current_device(&dev) == TPMLP_OK && dev) sms = dev->num_sms;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, 256, 0) != cudaSuccess || occ < 1) {
    cudaGetLastError();
    occ = 4;
  }
  const int64_t want = (units_per_chunk + 255) / 256;
  const int64_t per_chunk = std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(occ) * sms / nchunks));
  return dim3(static_cast<unsigned>(per_chunk), static_cast<unsigned>(nchunks));
}

template <int DT, int V>
bool ln_fwd_streamed_v(const ChunkSet& cs, const void* gamma, const void* beta, float eps, float* mean, float* rstd,
                       int64_t M, int64_t h, int64_t rpc, cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(ln_fwd_stream_kernel<DT, V>);
  const size_t rb = pad128(static_cast<uint32_t>(h * sizeof(typename Storage<DT>::T)));
  const StreamPlan p = plan_stream(fn, 2 * rb, rb, 3, M);
  if (!p.ok) return false;
  DeviceInfo* dev = nullptr;
  current_device(&dev);
  ln_fwd_stream_kernel<DT, V><<<p.grid, STREAM_THREADS, p.smem, st>>>(cs, gamma, beta, eps, mean, rstd, M, h, rpc,
                                                                     p.S, dev->status, wait_timeout_ns());
  return true;
}

template <int DT>
bool ln_fwd_streamed(const ChunkSet& cs, const void* gamma, const void* beta, float eps, float* mean, float* rstd,
                     int64_t M, int64_t h, int64_t rpc, cudaStream_t st) {
  switch ((h / 8 + STREAM_THREADS - 1) / STREAM_THREADS) {
    case 1: return ln_fwd_streamed_v<DT, 1>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
    case 2: return ln_fwd_streamed_v<DT, 2>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
    case 3: return ln_fwd_streamed_v<DT, 3>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
    case 4: return ln_fwd_streamed_v<DT, 4>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
    default: return false;
  }
}

template <int DT, int V>
bool ln_bwd_streamed_v(const ChunkSet& cs, const void* gamma, const float* mean, const float* rstd, int accumulate,
                       float* dgamma, float* dbeta, float* part, int64_t max_parts, int64_t M, int64_t h, int64_t rpc,
                       cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(ln_bwd_stream_kernel<DT, V>);
  const size_t rb = pad128(static_cast<uint32_t>(h * sizeof(typename Storage<DT>::T)));
  const StreamPlan p = plan_stream(fn, rb, (accumulate ? 3 : 2) * rb, 2, std::min(M, max_parts));
  if (!p.ok) return false;
  DeviceInfo* dev = nullptr;
  current_device(&dev);
  ln_bwd_stream_kernel<DT, V><<<p.grid, STREAM_THREADS, p.smem, st>>>(cs, gamma, mean, rstd, accumulate, part, M, h,
                                                                     rpc, p.S, dev->status, wait_timeout_ns());
  ln_bwd_reduce_parts_kernel<<<static_cast<unsigned>((2 * h + 31) / 32), 256, 0, st>>>(part, dgamma, dbeta, h,
                                                                                       p.grid);
  return true;
}

template <int DT>
bool ln_bwd_streamed(const ChunkSet& cs, const void* gamma, const float* mean, const float* rstd, int accumulate,
                     float* dgamma, float* dbeta, float* part, int64_t max_parts, int64_t M, int64_t h, int64_t rpc,
                     cudaStream_t st) {
  switch ((h / 8 + STREAM_THREADS - 1) / STREAM_THREADS) {
#define LNBS(V) \
  case V: return ln_bwd_streamed_v<DT, V>(cs, gamma, mean, rstd, accumulate, dgamma, dbeta, part, max_parts, M, h, rpc, st)
    LNBS(1);
    LNBS(2);
    LNBS(3);
    LNBS(4);
#undef LNBS
    default: return false;
  }
}

}  // namespace

int launch_ln_forward(const void* const* x, const void* gamma, const void* beta, float eps, void* const* y,
                      float* mean, float* rstd, int64_t M, int64_t h, int64_t rpc, int nchunks, int dtype,
                      cudaStream_t st) {
  if (M <= 0) return TPMLP_OK;
  ChunkSet cs{};
  for (int j = 0; j < nchunks; ++j) {
    cs.in[j] = x[j];
    cs.out[j] = y[j];
  }
  const size_t e = dtype == DT_F32 ? 4 : 2;
  const bool vec = h % 8 == 0 && ((align_bits(x, nchunks) | align_bits(const_cast<const void* const*>(y), nchunks) |
                                   reinterpret_cast<uintptr_t>(gamma) | reinterpret_cast<uintptr_t>(beta)) %
                                  (8 * e)) == 0;
  const int ph = prof_begin(PROF_SP_REGION, st);
  bool streamed = false;
  if (vec && h >= STREAM_MIN_H && h <= 8 * STREAM_THREADS * STREAM_MAX_V) {
    if (dtype == DT_F32) streamed = ln_fwd_streamed<DT_F32>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
    else if (dtype == DT_F16) streamed = ln_fwd_streamed<DT_F16>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
    else streamed = ln_fwd_streamed<DT_BF16>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
  }
  if (!streamed) {
    const int grid = static_cast<int>((M + ROWS_PER_CTA - 1) / ROWS_PER_CTA);
#define LNF(D, V) ln_fwd_kernel<D, V><<<grid, 256, 0, st>>>(cs, gamma, beta, eps, mean, rstd, M, h, rpc)
    if (dtype == DT_F32) { if (vec) LNF(DT_F32, true); else LNF(DT_F32, false); }
    else if (dtype == DT_F16) { if (vec) LNF(DT_F16, true); else LNF(DT_F16, false); }
    else { if (vec) LNF(DT_BF16, true); else LNF(DT_BF16, false); }
#undef LNF
  }
  prof_end(ph, static_cast<double>(M) * h * e * 2 + 8.0 * M, st);
  return check_launch("LayerNorm forward");
}

int launch_ln_backward(const void* const* x, const void* gamma, const float* mean, const float* rstd,
                       const void* const* dy, void* const* dx, int accumulate, float* dgamma, float* dbeta,
                       float* part, int64_t M, int64_t h, int64_t rpc, int nchunks, int dtype, cudaStream_t st) {
  if (M <= 0) {
    cudaError_t e = cudaMemsetAsync(dgamma, 0, sizeof(float) * h, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dbeta, 0, sizeof(float) * h, st);
    return e == cudaSuccess ? TPMLP_OK : set_error(TPMLP_ERR_CUDA, std::string("memset: ") + cudaGetErrorString(e));
  }
  ChunkSet cs{};
  for (int j = 0; j < nchunks; ++j) {
    cs.in[j] = x[j];
    cs.in2[j] = dy[j];
    cs.out[j] = dx[j];
  }
  const size_t e = dtype == DT_F32 ? 4 : 2;
  const bool vec = h % 8 == 0 && ((align_bits(x, nchunks) | align_bits(dy, nchunks) |
                                   align_bits(const_cast<const void* const*>(dx), nchunks) |
                                   reinterpret_cast<uintptr_t>(gamma)) % (8 * e)) == 0;
  // algorithmic bytes: x, dy read, dx written (and read when accumulating),
  // mean/rstd read, dγ/dβ written
  const double bytes = static_cast<double>(M) * h * e * (accumulate ? 4 : 3) + 8.0 * M + 8.0 * h;
  const int ph = prof_begin(PROF_SP_REGION, st);
  // fused path: one streamed pass writes dx and per-CTA dγ/dβ partials (at most
  // ⌈M/8⌉ of them, the rows the workspace holds), then a fixed-order reduction
  if (vec && h >= STREAM_MIN_H && h <= 8 * STREAM_THREADS * STREAM_MAX_V) {
    const int64_t max_parts = (M + 7) / 8;
    bool streamed;
    if (dtype == DT_F32)
      streamed = ln_bwd_streamed<DT_F32>(cs, gamma, mean, rstd, accumulate, dgamma, dbeta, part, max_parts, M, h, rpc, st);
    else if (dtype == DT_F16)
      streamed = ln_bwd_streamed<DT_F16>(cs, gamma, mean, rstd, accumulate, dgamma, dbeta, part, max_parts, M, h, rpc, st);
    else
      streamed = ln_bwd_streamed<DT_BF16>(cs, gamma, mean, rstd, accumulate, dgamma, dbeta, part, max_parts, M, h, rpc, st);
    if (streamed) {
      prof_end(ph, bytes, st, 2);
      return check_launch("LayerNorm backward");
    }
  }
  // warp-per-row pass for dx, then a column pass for the dγ/dβ partials
  const int grid = static_cast<int>((M + ROWS_PER_CTA - 1) / ROWS_PER_CTA);
#define LNB(D, V) ln_bwd_rows_kernel<D, V><<<grid, 256, 0, st>>>(cs, gamma, mean, rstd, accumulate, M, h, rpc)
  if (dtype == DT_F32) { if (vec) LNB(DT_F32, true); else LNB(DT_F32, false); }
  else if (dtype == DT_F16) { if (vec) LNB(DT_F16, true); else LNB(DT_F16, false); }
  else { if (vec) LNB(DT_BF16, true); else LNB(DT_BF16, false); }
#undef LNB
  const int rc = check_launch("LayerNorm backward (rows)");
  if (rc != TPMLP_OK) return rc;
  if (vec) {
    // vectorised column pass: 8 columns per thread, 16-token blocks
    const int64_t nrb_v = (M + VCOL_ROWS - 1) / VCOL_ROWS;
    dim3 g2(static_cast<unsigned>((h / 8 + 255) / 256), static_cast<unsigned>(nrb_v));
    if (dtype == DT_F32) ln_bwd_cols_vec_kernel<DT_F32><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb_v);
    else if (dtype == DT_F16) ln_bwd_cols_vec_kernel<DT_F16><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb_v);
    else ln_bwd_cols_vec_kernel<DT_BF16><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb_v);
    ln_bwd_reduce_kernel<<<static_cast<unsigned>((h + 255) / 256), 256, 0, st>>>(part, dgamma, dbeta, h, nrb_v);
  } else {
    const int64_t nrb = (M + COL_ROWS - 1) / COL_ROWS;
    dim3 g2(static_cast<unsigned>((h + 255) / 256), static_cast<unsigned>(nrb));
    if (dtype == DT_F32) ln_bwd_cols_kernel<DT_F32><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb);
    else if (dtype == DT_F16) ln_bwd_cols_kernel<DT_F16><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb);
    else ln_bwd_cols_kernel<DT_BF16><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb);
    ln_bwd_reduce_kernel<<<static_cast<unsigned>((h + 255) / 256), 256, 0, st>>>(part, dgamma, dbeta, h, nrb);
  }
  prof_end(ph, bytes, st, 3);
  return check_launch("LayerNorm backward (gamma, beta)");
}

int launch_residual_dropout(bool forward, const void* const* r, const void* const* z, const uint8_t* const* keep,
                            float p, void* const* out, int64_t n_chunk, int nchunks, int dtype, cudaStream_t st) {
  if (n_chunk <= 0) return TPMLP_OK;
  ChunkSet cs{};
  for (int j = 0; j < nchunks; ++j) {
    cs.in[j] = forward ? r[j] : nullptr;
    cs.in2[j] = z[j];
    cs.mask[j] = keep[j];
    cs.out[j] = out[j];
  }
  const float scale = 1.0f / (1.0f - p);
  const size_t e = dtype == DT_F32 ? 4 : 2;
  uintptr_t al = align_bits(z, nchunks) | align_bits(const_cast<const void* const*>(out), nchunks);
  if (forward) al |= align_bits(r, nchunks);
  const bool vec = n_chunk % 8 == 0 && (al % (8 * e)) == 0 &&
                   (align_bits(reinterpret_cast<const void* const*>(keep), nchunks) % 8) == 0;
  const int ph = prof_begin(PROF_SP_REGION, st);
#define RD(D, F)                                                                                         \
  do {                                                                                                   \
    if (vec) {                                                                                           \
      const dim3 g = dropout_grid(reinterpret_cast<const void*>(residual_dropout_vec8_kernel<D, F>),      \
                                  n_chunk / 32, nchunks);                                                \
      residual_dropout_vec8_kernel<D, F><<<g, 256, 0, st>>>(cs, scale, n_chunk);                         \
    } else {                                                                                             \
      const dim3 g = dropout_grid(reinterpret_cast<const void*>(residual_dropout_kernel<D, F>), n_chunk,   \
                                  nchunks);                                                              \
      residual_dropout_kernel<D, F><<<g, 256, 0, st>>>(cs, scale, n_chunk);                              \
    }                                                                                                    \
  } while (0)
  if (forward) {
    if (dtype == DT_F32) RD(DT_F32, true); else if (dtype == DT_F16) RD(DT_F16, true); else RD(DT_BF16, true);
  } else {
    if (dtype == DT_F32) RD(DT_F32, false); else if (dtype == DT_F16) RD(DT_F16, false); else RD(DT_BF16, false);
  }
#undef RD
  prof_end(ph, static_cast<double>(n_chunk) * nchunks * (e * (forward ? 3 : 2) + 1), st);
  return check_launch("residual dropout");
}

}  // namespace tpmlp

// ---------------------------------------------------------------- C ABI
using namespace tpmlp;

namespace {

int check_region(int64_t s, int64_t b, int64_t h, int tp, int dtype) {
  if (s < 0 || b < 0 || h <= 0) return set_error(TPMLP_ERR_INVALID_ARG, "s, b >= 0 and h >= 1 required");
  if (tp < 1 || tp > TPMLP_MAX_TP) return set_error(TPMLP_ERR_INVALID_ARG, "tp must be in [1, 64]");
  if (dtype < DT_F32 || dtype > DT_BF16) return set_error(TPMLP_ERR_INVALID_ARG, "unknown dtype");
  if (s * b >= (1ll << 31) || h >= (1ll << 31)) return set_error(TPMLP_ERR_UNSUPPORTED, "extent too large");
  if (s % tp != 0)
    return set_error(TPMLP_ERR_NOT_DIVISIBLE, "First dimension of the tensor should be divisible by tensor parallel size");
  return TPMLP_OK;
}

int check_arr(const void* const* a, int n, size_t align, const char* name) {
  if (a == nullptr) return set_error(TPMLP_ERR_INVALID_ARG, std::string(name) + " array is NULL");
  for (int i = 0; i < n; ++i) {
    if (a[i] == nullptr) return set_error(TPMLP_ERR_INVALID_ARG, std::string(name) + " is NULL");
    if (reinterpret_cast<uintptr_t>(a[i]) % align != 0)
      return set_error(TPMLP_ERR_INVALID_ARG, std::string(name) + " is misaligned");
  }
  return TPMLP_OK;
}

int check_one(const void* p, size_t align, const char* name) { return check_arr(&p, 1, align, name); }

size_t esize(int dtype) { return dtype == DT_F32 ? 4 : 2; }

}  // namespace

extern "C" {

int tpmlp_sp_layernorm_forward(const void* const* x, const void* gamma, const void* beta, float eps, void* const* y,
                               float* mean, float* rstd, int64_t s, int64_t b, int64_t h, int tp, int dtype,
                               void* stream) {
  int rc = check_region(s, b, h, tp, dtype);
  if (rc) return rc;
  if (!(eps >= 0.0f)) return set_error(TPMLP_ERR_INVALID_ARG, "eps must be >= 0");
  const size_t e = esize(dtype);
  if ((rc = check_arr(x, tp, e, "x")) || (rc = check_arr(const_cast<const void* const*>(y), tp, e, "y")) ||
      (rc = check_one(gamma, e, "gamma")) || (rc = check_one(beta, e, "beta")) || (rc = check_one(mean, 4, "mean")) ||
      (rc = check_one(rstd, 4, "rstd")))
    return rc;
  return launch_ln_forward(x, gamma, beta, eps, y, mean, rstd, s * b, h, (s / tp) * b, tp, dtype,
                           static_cast<cudaStream_t>(stream));
}

size_t tpmlp_sp_layernorm_backward_workspace(int64_t s, int64_t b, int64_t h) {
  if (s < 0 || b < 0 || h <= 0) return 0;
  // up to ⌈s·b/8⌉ partial rows for each of dγ and dβ (one per CTA of the streamed
  // pass, or one per 16- or 128-token block of the column pass)
  const int64_t nrb = (s * b + 7) / 8;
  return static_cast<size_t>(2 * nrb * h) * sizeof(float);
}

int tpmlp_sp_layernorm_backward(const void* const* x, const void* gamma, const float* mean, const float* rstd,
                                const void* const* dy, void* const* dx, int accumulate, float* dgamma, float* dbeta,
                                void* ws, size_t ws_bytes, int64_t s, int64_t b, int64_t h, int tp, int dtype,
                                void* stream) {
  int rc = check_region(s, b, h, tp, dtype);
  if (rc) return rc;
  if (accumulate != 0 && accumulate != 1) return set_error(TPMLP_ERR_INVALID_ARG, "accumulate must be 0 or 1");
  const size_t e = esize(dtype);
  if ((rc = check_arr(x, tp, e, "x")) || (rc = check_arr(dy, tp, e, "dy")) ||
      (rc = check_arr(const_cast<const void* const*>(dx), tp, e, "dx")) || (rc = check_one(gamma, e, "gamma")) ||
      (rc = check_one(mean, 4, "mean")) || (rc = check_one(rstd, 4, "rstd")) || (rc = check_one(dgamma, 4, "dgamma")) ||
      (rc = check_one(dbeta, 4, "dbeta")))
    return rc;
  const size_t need = tpmlp_sp_layernorm_backward_workspace(s, b, h);
  if (need > 0 && (ws == nullptr || ws_bytes < need))
    return set_error(TPMLP_ERR_WORKSPACE, "LayerNorm backward workspace needs " + std::to_string(need) + " bytes");
  if (need > 0 && (rc = check_one(ws, 16, "ws"))) return rc;
  return launch_ln_backward(x, gamma, mean, rstd, dy, dx, accumulate, dgamma, dbeta, static_cast<float*>(ws), s * b,
                            h, (s / tp) * b, tp, dtype, static_cast<cudaStream_t>(stream));
}

int tpmlp_sp_residual_dropout_forward(const void* const* r, const void* const* z, const uint8_t* const* keep, float p,
                                      void* const* out, int64_t s, int64_t b, int64_t h, int tp, int dtype,
                                      void* stream) {
  int rc = check_region(s, b, h, tp, dtype);
  if (rc) return rc;
  if (!(p >= 0.0f && p < 1.0f)) return set_error(TPMLP_ERR_INVALID_ARG, "dropout probability must be in [0, 1)");
  const size_t e = esize(dtype);
  if ((rc = check_arr(r, tp, e, "r")) || (rc = check_arr(z, tp, e, "z")) ||
      (rc = check_arr(reinterpret_cast<const void* const*>(keep), tp, 1, "keep")) ||
      (rc = check_arr(const_cast<const void* const*>(out), tp, e, "out")))
    return rc;
  return launch_residual_dropout(true, r, z, keep, p, out, (s / tp) * b * h, tp, dtype,
                                 static_cast<cudaStream_t>(stream));
}

int tpmlp_sp_residual_dropout_backward(const void* const* dout, const uint8_t* const* keep, float p, void* const* dz,
                                       int64_t s, int64_t b, int64_t h, int tp, int dtype, void* stream) {
  int rc = check_region(s, b, h, tp, dtype);
  if (rc) return rc;
  if (!(p >= 0.0f && p < 1.0f)) return set_error(TPMLP_ERR_INVALID_ARG, "dropout probability must be in [0, 1)");
  const size_t e = esize(dtype);
  if ((rc = check_arr(dout, tp, e, "dout")) ||
      (rc = check_arr(reinterpret_cast<const void* const*>(keep), tp, 1, "keep")) ||
      (rc = check_arr(const_cast<const void* const*>(dz), tp, e, "dz")))
    return rc;
  return launch_residual_dropout(false, nullptr, dout, keep, p, dz, (s / tp) * b * h, tp, dtype,
                                 static_cast<cudaStream_t>(stream));
}

}  // extern "C"
