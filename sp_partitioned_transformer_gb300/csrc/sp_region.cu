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
//   ln_fwd_kernel         one warp per token: mean, variance (two passes over the
//                         row, re-read from L1), normalise + affine, save mean/rstd;
//   ln_bwd_rows_kernel    one warp per token: dx = rstd·(g − mean(g) − x̂·mean(g·x̂)),
//                         g = dy·γ, written or added to the residual gradient;
//   ln_bwd_cols_kernel    dγ, dβ partial sums over 128-token blocks (coalesced
//                         along h), then ln_bwd_reduce_kernel adds the blocks in a
//                         fixed order: deterministic parameter gradients;
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

// ------------------------------------------------------------------ row-resident variants
// One CTA of 256 threads per token row, the row held in registers (up to
// RV vectors of 8 elements per thread: h <= 8192), block-wide reductions: every
// load of the row is in flight at once and the row is read from HBM once.
constexpr int RV = 4;

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // previous use of red[] finished
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = lane < (blockDim.x >> 5) ? red[lane] : 0.0f;
  return warp_sum(t);
}

// The row stays packed in its storage type (16 registers for 32 bf16 values per
// thread) so that four or more CTAs fit per SM: enough bytes in flight.
template <int DT>
struct Packed8 {
  uint4 w[DT == DT_F32 ? 2 : 1];
  __device__ __forceinline__ void load(const void* p, int64_t i) {
    if constexpr (DT == DT_F32) {
      w[0] = *reinterpret_cast<const uint4*>(static_cast<const float*>(p) + i);
      w[1] = *reinterpret_cast<const uint4*>(static_cast<const float*>(p) + i + 4);
    } else {
      w[0] = *reinterpret_cast<const uint4*>(static_cast<const typename Storage<DT>::T*>(p) + i);
    }
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

template <int DT>
__global__ void __launch_bounds__(256, 4) ln_fwd_row_kernel(ChunkSet cs, const void* __restrict__ gamma,
                                                            const void* __restrict__ beta, float eps,
                                                            float* __restrict__ mean, float* __restrict__ rstd,
                                                            int64_t h, int64_t rpc) {
  __shared__ float red[8];
  const int64_t m = blockIdx.x;
  const int64_t j = m / rpc;
  const int64_t off = (m - j * rpc) * h;
  const void* x = cs.in[j];
  void* y = cs.out[j];
  const int nv = static_cast<int>(h / 8);
  Packed8<DT> raw[RV];
#pragma unroll
  for (int k = 0; k < RV; ++k)
    if (threadIdx.x + k * 256 < nv) raw[k].load(x, off + (threadIdx.x + k * 256) * 8);
  float sum = 0.0f;
#pragma unroll
  for (int k = 0; k < RV; ++k)
    if (threadIdx.x + k * 256 < nv) {
      float v[8];
      raw[k].unpack(v);
#pragma unroll
      for (int i = 0; i < 8; ++i) sum += v[i];
    }
  const float inv_h = 1.0f / static_cast<float>(h);
  const float mu = block_sum(sum, red) * inv_h;
  float q = 0.0f;
#pragma unroll
  for (int k = 0; k < RV; ++k)
    if (threadIdx.x + k * 256 < nv) {
      float v[8];
      raw[k].unpack(v);
#pragma unroll
      for (int i = 0; i < 8; ++i) q += (v[i] - mu) * (v[i] - mu);
    }
  const float r = 1.0f / sqrtf(block_sum(q, red) * inv_h + eps);
#pragma unroll
  for (int k = 0; k < RV; ++k) {
    const int vi = threadIdx.x + k * 256;
    if (vi < nv) {
      float v[8], g[8], b[8], o[8];
      raw[k].unpack(v);
      ld8<DT>(gamma, vi * 8, g);
      ld8<DT>(beta, vi * 8, b);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = (v[i] - mu) * r * g[i] + b[i];
      st8<DT>(y, off + vi * 8, o);
    }
  }
  if (threadIdx.x == 0) {
    mean[m] = mu;
    rstd[m] = r;
  }
}

template <int DT>
__global__ void __launch_bounds__(256, 3) ln_bwd_row_kernel(ChunkSet cs, const void* __restrict__ gamma,
                                                            const float* __restrict__ mean,
                                                            const float* __restrict__ rstd, int accumulate, int64_t h,
                                                            int64_t rpc) {
  __shared__ float red[8];
  const int64_t m = blockIdx.x;
  const int64_t j = m / rpc;
  const int64_t off = (m - j * rpc) * h;
  const void* x = cs.in[j];
  const void* dy = cs.in2[j];
  void* dx = cs.out[j];
  const float mu = mean[m], r = rstd[m];
  const int nv = static_cast<int>(h / 8);
  Packed8<DT> rx[RV], rd[RV];
#pragma unroll
  for (int k = 0; k < RV; ++k)
    if (threadIdx.x + k * 256 < nv) {
      rx[k].load(x, off + (threadIdx.x + k * 256) * 8);
      rd[k].load(dy, off + (threadIdx.x + k * 256) * 8);
    }
  float sg = 0.0f, sgx = 0.0f;
#pragma unroll
  for (int k = 0; k < RV; ++k) {
    const int vi = threadIdx.x + k * 256;
    if (vi < nv) {
      float xv[8], d[8], g[8];
      rx[k].unpack(xv);
      rd[k].unpack(d);
      ld8<DT>(gamma, vi * 8, g);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float gi = d[i] * g[i];
        sg += gi;
        sgx += gi * (xv[i] - mu) * r;
      }
    }
  }
  const float inv_h = 1.0f / static_cast<float>(h);
  const float mg = block_sum(sg, red) * inv_h;
  const float mgx = block_sum(sgx, red) * inv_h;
#pragma unroll
  for (int k = 0; k < RV; ++k) {
    const int vi = threadIdx.x + k * 256;
    if (vi < nv) {
      float xv[8], d[8], g[8], o[8];
      rx[k].unpack(xv);
      rd[k].unpack(d);
      ld8<DT>(gamma, vi * 8, g);
      if (accumulate) ld8<DT>(dx, off + vi * 8, o);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float t = r * (d[i] * g[i] - mg - (xv[i] - mu) * r * mgx);
        o[i] = accumulate ? o[i] + t : t;
      }
      st8<DT>(dx, off + vi * 8, o);
    }
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

template <int DT, bool FWD>
__global__ void __launch_bounds__(256) residual_dropout_vec8_kernel(ChunkSet cs, float scale, int64_t n_chunk) {
  constexpr int U = 4;  // vectors of 8 elements in flight per thread
  const int j = blockIdx.y;
  const uint8_t* keep = static_cast<const uint8_t*>(cs.mask[j]);
  const int64_t nvec = n_chunk / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t v0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v0 < nvec; v0 += U * stride) {
    float z[U][8], r[U][8];
    uint2 k8[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nvec) {
        ld8<DT>(cs.in2[j], v * 8, z[u]);
        if (FWD) ld8<DT>(cs.in[j], v * 8, r[u]);
        k8[u] = *reinterpret_cast<const uint2*>(keep + v * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nvec) {
        const uint8_t* kb = reinterpret_cast<const uint8_t*>(&k8[u]);
        float o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float kz = kb[i] ? z[u][i] * scale : 0.0f;
          o[i] = FWD ? r[u][i] + kz : kz;
        }
        st8<DT>(cs.out[j], v * 8, o);
      }
    }
  }
}

int grid_1d(int64_t work_items, int64_t per_cta) {
  DeviceInfo* dev = nullptr;
  int sms = 148;
  if (current_device(&dev) == TPMLP_OK && dev) sms = dev->num_sms;
  const int64_t want = (work_items + per_cta - 1) / per_cta;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(sms) * 8)));
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
  const int grid = static_cast<int>((M + ROWS_PER_CTA - 1) / ROWS_PER_CTA);
  const int ph = prof_begin(PROF_SP_REGION, st);
  if (vec && h <= 256 * 8 * RV) {
    const unsigned rows = static_cast<unsigned>(M);
    if (dtype == DT_F32) ln_fwd_row_kernel<DT_F32><<<rows, 256, 0, st>>>(cs, gamma, beta, eps, mean, rstd, h, rpc);
    else if (dtype == DT_F16) ln_fwd_row_kernel<DT_F16><<<rows, 256, 0, st>>>(cs, gamma, beta, eps, mean, rstd, h, rpc);
    else ln_fwd_row_kernel<DT_BF16><<<rows, 256, 0, st>>>(cs, gamma, beta, eps, mean, rstd, h, rpc);
  } else {
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
  const int64_t nrb = (M + COL_ROWS - 1) / COL_ROWS;
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
  const int grid = static_cast<int>((M + ROWS_PER_CTA - 1) / ROWS_PER_CTA);
  const bool row_resident = vec && h <= 256 * 8 * RV;
  int ph = prof_begin(PROF_SP_REGION, st);
  if (row_resident) {
    const unsigned rows = static_cast<unsigned>(M);
    if (dtype == DT_F32) ln_bwd_row_kernel<DT_F32><<<rows, 256, 0, st>>>(cs, gamma, mean, rstd, accumulate, h, rpc);
    else if (dtype == DT_F16) ln_bwd_row_kernel<DT_F16><<<rows, 256, 0, st>>>(cs, gamma, mean, rstd, accumulate, h, rpc);
    else ln_bwd_row_kernel<DT_BF16><<<rows, 256, 0, st>>>(cs, gamma, mean, rstd, accumulate, h, rpc);
  } else {
#define LNB(D, V) ln_bwd_rows_kernel<D, V><<<grid, 256, 0, st>>>(cs, gamma, mean, rstd, accumulate, M, h, rpc)
    if (dtype == DT_F32) { if (vec) LNB(DT_F32, true); else LNB(DT_F32, false); }
    else if (dtype == DT_F16) { if (vec) LNB(DT_F16, true); else LNB(DT_F16, false); }
    else { if (vec) LNB(DT_BF16, true); else LNB(DT_BF16, false); }
#undef LNB
  }
  prof_end(ph, static_cast<double>(M) * h * e * (accumulate ? 4 : 3) + 8.0 * M, st);
  int rc = check_launch("LayerNorm backward (rows)");
  if (rc != TPMLP_OK) return rc;
  ph = prof_begin(PROF_SP_REGION, st);
  if (vec) {
    // vectorised column pass: 8 columns per thread, 32-token blocks
    const int64_t nrb_v = (M + VCOL_ROWS - 1) / VCOL_ROWS;
    dim3 g2(static_cast<unsigned>((h / 8 + 255) / 256), static_cast<unsigned>(nrb_v));
    if (dtype == DT_F32) ln_bwd_cols_vec_kernel<DT_F32><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb_v);
    else if (dtype == DT_F16) ln_bwd_cols_vec_kernel<DT_F16><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb_v);
    else ln_bwd_cols_vec_kernel<DT_BF16><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb_v);
    ln_bwd_reduce_kernel<<<static_cast<unsigned>((h + 255) / 256), 256, 0, st>>>(part, dgamma, dbeta, h, nrb_v);
    prof_end(ph, static_cast<double>(M) * h * e * 2 + 16.0 * nrb_v * h, st);
  } else {
    dim3 g2(static_cast<unsigned>((h + 255) / 256), static_cast<unsigned>(nrb));
    if (dtype == DT_F32) ln_bwd_cols_kernel<DT_F32><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb);
    else if (dtype == DT_F16) ln_bwd_cols_kernel<DT_F16><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb);
    else ln_bwd_cols_kernel<DT_BF16><<<g2, 256, 0, st>>>(cs, mean, rstd, part, M, h, rpc, nrb);
    ln_bwd_reduce_kernel<<<static_cast<unsigned>((h + 255) / 256), 256, 0, st>>>(part, dgamma, dbeta, h, nrb);
    prof_end(ph, static_cast<double>(M) * h * e * 2 + 16.0 * nrb * h, st);
  }
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
  // about 8 CTAs per SM in total over the nchunks rows of the grid (the vector
  // kernel handles four 8-element vectors per thread per iteration)
  const int per_chunk = std::max(1, grid_1d(vec ? n_chunk / 32 : n_chunk, 256) / nchunks);
  dim3 grid(static_cast<unsigned>(per_chunk), static_cast<unsigned>(nchunks));
  const int ph = prof_begin(PROF_SP_REGION, st);
#define RD(D, F)                                                                        \
  do {                                                                                  \
    if (vec) residual_dropout_vec8_kernel<D, F><<<grid, 256, 0, st>>>(cs, scale, n_chunk); \
    else residual_dropout_kernel<D, F><<<grid, 256, 0, st>>>(cs, scale, n_chunk);          \
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
  const int64_t nrb = (s * b + 15) / 16;  // 16-token partial blocks (the 128-token variant needs less)
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
