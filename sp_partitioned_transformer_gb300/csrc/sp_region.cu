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
//   ln_fwd_pair_kernel    16-bit rows of an even number of vectors, 2k < h/8 ≤ 8k
//                         (h up to 8192): two warps per row sharing one TMA-filled slot, each
//                         holding half the row in registers, their shifted sums
//                         combined through shared memory;
//   ln_fwd_warp_kernel    other 16-bit rows up to h = 8192: one warp per row, each
//                         warp's row brought in by TMA bulk copies into its own
//                         slot and held in registers; one-pass shifted
//                         statistics, normalise + affine, save mean/rstd;
//   ln_fwd_stream_kernel  float32 rows (h >= 1024, 16-byte aligned): persistent
//                         CTAs stream rows through a TMA-bulk shared-memory ring;
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

// ------------------------------------------------------------------ rows held in registers
// 16-bit rows up to h = 8192 as NV 8-element vectors a lane (lane l owns the
// vectors l, l + 32, …), kept packed: at most 128 data registers a thread.
constexpr int REG_MAX_NV = 32;

// 8 packed 16-bit values -> 4 float pairs (a bf16 is the upper half of the
// float with the same value: one shift and one mask per pair).
template <int DT>
__device__ __forceinline__ void unpack8_pairs(const uint4& r, float2* f) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (DT == DT_BF16)
      f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    else
      f[i] = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
  }
}

// The same conversion as volatile asm: the compiler converts again at every
// use and cannot hoist conversions ahead, which keeps the backward's registers
// (row vectors, dγ/dβ accumulators) within two CTAs per SM.
template <int DT>
__device__ __forceinline__ void unpack8_pairs_v(const uint4& r, float2* f) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (DT == DT_BF16) {
      // a bf16 is the upper half of the float with the same value
      uint32_t lo, hi;
      asm volatile("{\n\tshl.b32 %0, %2, 16;\n\tand.b32 %1, %2, 0xffff0000;\n\t}" : "=r"(lo), "=r"(hi) : "r"(w[i]));
      f[i] = make_float2(__uint_as_float(lo), __uint_as_float(hi));
    } else {
      float a, b;
      asm volatile("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
                   : "=f"(a), "=f"(b)
                   : "r"(w[i]));
      f[i] = make_float2(a, b);
    }
  }
}

// A 16-byte shared-memory load issued where it stands (volatile: not hoisted
// ahead of the loop that uses it, which would hold every vector's γ and β in
// registers at once).
__device__ __forceinline__ uint4 lds_v4(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// y = x·γ + β on 8 packed 16-bit values, two per fused multiply-add.
template <int DT>
__device__ __forceinline__ uint4 affine8_packed(const uint4& x, const uint4& g, const uint4& b) {
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, gw[4] = {g.x, g.y, g.z, g.w}, bw[4] = {b.x, b.y, b.z, b.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (DT == DT_BF16) {
      const __nv_bfloat162 r = __hfma2(*reinterpret_cast<const __nv_bfloat162*>(&xw[i]),
                                       *reinterpret_cast<const __nv_bfloat162*>(&gw[i]),
                                       *reinterpret_cast<const __nv_bfloat162*>(&bw[i]));
      o[i] = *reinterpret_cast<const uint32_t*>(&r);
    } else {
      const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&xw[i]), *reinterpret_cast<const __half2*>(&gw[i]),
                                *reinterpret_cast<const __half2*>(&bw[i]));
      o[i] = *reinterpret_cast<const uint32_t*>(&r);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// An optimisation barrier on a row held in registers: the compiler must assume
// the packed values changed, so it converts them again at their next use
// instead of keeping every converted float of the row live (which would double
// the registers a row needs).  It emits no instruction.
template <int NV>
__device__ __forceinline__ void reg_fence(uint4 (&v)[NV]) {
#pragma unroll
  for (int k = 0; k < NV; ++k) asm volatile("" : "+r"(v[k].x), "+r"(v[k].y), "+r"(v[k].z), "+r"(v[k].w));
}

template <int DT>
__device__ __forceinline__ uint4 pack8_pairs(const float2* f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (DT == DT_BF16) {
      const __nv_bfloat162 b = __float22bfloat162_rn(f[i]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    } else {
      const __half2 b = __float22half2_rn(f[i]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
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
template <int THREADS = STREAM_THREADS>
__device__ __forceinline__ float2 block_sum2_free(float a, float b, float2* red) {
  a = warp_sum(a);
  b = warp_sum(b);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[w] = make_float2(a, b);
  __syncthreads();
  const float2 t = lane < THREADS / 32 ? red[lane] : make_float2(0.0f, 0.0f);
  return make_float2(warp_sum(t.x), warp_sum(t.y));
}

struct RowRing {
  uint8_t* base;   // slot 0
  uint32_t rb;     // bytes of one row
  uint32_t rb_al;  // ... padded to 128
  int nin;         // rows per slot
  int S;           // slots
};

// Where row m = m0 + k·G lies, as (chunk j, row r of the chunk), stepped from
// one k to the next without a division (G = qG·rpc + rG): a 64-bit division
// is a long software sequence on the GPU, and these kernels advance a row at a
// time.
struct RowStep {
  int64_t qG, rG, rpc;
  __device__ __forceinline__ RowStep(int64_t G, int64_t rpc_) : qG(G / rpc_), rG(G - (G / rpc_) * rpc_), rpc(rpc_) {}
};
struct RowPos {
  int64_t j, r;
  __device__ __forceinline__ RowPos(int64_t m0, const RowStep& st) : j(m0 / st.rpc), r(m0 - (m0 / st.rpc) * st.rpc) {}
  __device__ __forceinline__ void next(const RowStep& st) {
    j += st.qG;
    r += st.rG;
    if (r >= st.rpc) {
      r -= st.rpc;
      ++j;
    }
  }
};

// Thread 0: start the bulk copies of the row at `pos` into slot s.
__device__ __forceinline__ void ring_issue(const RowRing& ring, uint64_t* full, const ChunkSet& cs, int s,
                                          const RowPos& pos, int64_t h, size_t esz) {
  const int64_t j = pos.j;
  const int64_t off = pos.r * h * static_cast<int64_t>(esz);
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

// ------------------------------------------------------------------ LN forward, one warp per row
// Persistent CTAs of `wpc` warps, one per SM.  Warp w of CTA c takes the rows
// g, g + W, g + 2W, … (g = c·wpc + w, W = all warps of the grid).  Each warp
// owns one shared-memory slot: a TMA bulk copy (issued by lane 0) brings row k
// into it, the lanes copy the row into registers (NV packed vectors a lane) and
// at once lane 0 refills the slot with row k + 1, whose load then overlaps row
// k's arithmetic.  γ and β are staged in shared memory once per CTA (the only
// block barrier).  Statistics take one pass over the registers: the shifted
// sums Σ(x − c), Σ(x − c)² with c the row's first element (which keeps the
// variance when the mean is large against the spread) in two independent pairs
// of accumulators, both warp reductions interleaved; then y = x̂·γ + β with
// x̂ = (x − μ)·rstd computed in float32 and rounded once to the storage type,
// the affine step a packed 16-bit fused multiply-add (one more rounding of the
// storage type's order than an all-float32 evaluation).  EXACT: every lane owns
// exactly NV vectors (h = 256·NV) and no vector is predicated.
template <int NV>
struct LnFwdShape {
  static constexpr int MAX_WARPS = NV <= 24 ? 16 : 8;  // registers: 128 (NV ≤ 24) or 255 a thread
};

template <int DT, int NV, bool EXACT>
__global__ void __launch_bounds__(32 * LnFwdShape<NV>::MAX_WARPS, 1)
    ln_fwd_warp_kernel(ChunkSet cs, const void* __restrict__ gamma, const void* __restrict__ beta, float eps,
                       float* __restrict__ mean, float* __restrict__ rstd, int64_t M, int64_t h, int64_t rpc,
                       unsigned* status, uint64_t timeout_ns) {
  static_assert(DT != DT_F32 && NV >= 1 && NV <= REG_MAX_NV, "16-bit rows of at most 32 vectors a lane");
  using T = typename Storage<DT>::T;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[LnFwdShape<NV>::MAX_WARPS];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int wpc = blockDim.x >> 5;
  const int nv = static_cast<int>(h / 8);
  const uint32_t rb = static_cast<uint32_t>(h * sizeof(T));
  uint4* gs = reinterpret_cast<uint4*>(smem);  // γ, β (16-bit, as stored)
  uint4* bs = reinterpret_cast<uint4*>(smem + pad128(rb));
  uint8_t* slot = smem + 2 * pad128(rb) + static_cast<size_t>(w) * pad128(rb);
  const uint32_t bar = smem_u32(&full[w]);
  const int64_t W = static_cast<int64_t>(gridDim.x) * wpc;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * wpc + w;
  const int64_t cnt = g < M ? (M - g + W - 1) / W : 0;
  const RowStep step(W, rpc);
  RowPos cur(g, step);  // the row computed
  auto issue = [&](const RowPos& at) {  // lane 0: the row at `at` into the slot
    mbar_arrive_expect_tx(bar, rb);
    bulk_g2s(smem_u32(slot), static_cast<const uint8_t*>(cs.in[at.j]) + at.r * h * static_cast<int64_t>(sizeof(T)),
             rb, bar);
  };
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    if (cnt > 0) issue(cur);
  }
  for (int vi = threadIdx.x; vi < nv; vi += blockDim.x) {
    gs[vi] = __ldg(static_cast<const uint4*>(gamma) + vi);
    bs[vi] = __ldg(static_cast<const uint4*>(beta) + vi);
  }
  __syncthreads();
  const float inv_h = 1.0f / static_cast<float>(h);
  for (int64_t k = 0; k < cnt; ++k) {
    // every lane waits (acquiring the bulk copy's bytes itself); all give up together
    const bool ok = mbar_wait_bounded(bar, static_cast<uint32_t>(k & 1), nullptr, status, timeout_ns);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) (void)mbar_wait_bounded(bar, static_cast<uint32_t>(k & 1), nullptr, nullptr, timeout_ns);
      return;
    }
    uint4 v[NV];
    const uint4* row = reinterpret_cast<const uint4*>(slot);
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      const int vi = lane + 32 * kk;
      v[kk] = (EXACT || vi < nv) ? row[vi] : make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();  // every lane has copied the row out of the slot
    if (lane == 0 && k + 1 < cnt) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      RowPos at = cur;
      at.next(step);
      issue(at);
    }
    // c = the row's first element (lane 0's first value)
    float c;
    {
      float2 f0[4];
      unpack8_pairs<DT>(v[0], f0);
      c = __shfl_sync(0xffffffffu, f0[0].x, 0);
    }
    const float2 nc2 = make_float2(-c, -c);
    // two independent pairs of accumulators (for the even and the odd float
    // pairs of a vector): the sums' dependency chains are half as long
    float2 s1[2], s2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) s1[i] = s2[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      if (EXACT || lane + 32 * kk < nv) {
        float2 f[4];
        unpack8_pairs<DT>(v[kk], f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 d = __fadd2_rn(f[i], nc2);
          s1[i & 1] = __fadd2_rn(s1[i & 1], d);
          s2[i & 1] = __ffma2_rn(d, d, s2[i & 1]);
        }
      }
    }
    const float2 t1 = __fadd2_rn(s1[0], s1[1]);
    const float2 t2 = __fadd2_rn(s2[0], s2[1]);
    float q1 = t1.x + t1.y, q2 = t2.x + t2.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {  // both warp sums, interleaved
      q1 += __shfl_xor_sync(0xffffffffu, q1, o);
      q2 += __shfl_xor_sync(0xffffffffu, q2, o);
    }
    const float dm = q1 * inv_h;
    const float var = fmaxf(q2 * inv_h - dm * dm, 0.0f);
    const float mu = c + dm;
    const float r = 1.0f / sqrtf(var + eps);
    reg_fence(v);
    // y = (x·r − μ·r)·γ + β
    const float2 r2 = make_float2(r, r);
    const float2 nmr2 = make_float2(-mu * r, -mu * r);
    const int64_t m = g + k * W;
    uint4* y = reinterpret_cast<uint4*>(static_cast<T*>(cs.out[cur.j]) + cur.r * h);
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      const int vi = lane + 32 * kk;
      if (EXACT || vi < nv) {
        // x̂ = (x − μ)·rstd in float32, rounded once to 16 bits; y = x̂·γ + β as
        // one packed 16-bit fused multiply-add (a single rounding of the result)
        float2 f[4], xh[4];
        unpack8_pairs<DT>(v[kk], f);
#pragma unroll
        for (int i = 0; i < 4; ++i) xh[i] = __ffma2_rn(f[i], r2, nmr2);
        y[vi] = affine8_packed<DT>(pack8_pairs<DT>(xh), lds_v4(gs + vi), lds_v4(bs + vi));
      }
    }
    if (lane == 0) {
      mean[m] = mu;
      rstd[m] = r;
    }
    cur.next(step);
  }
}

// Two warps per row: warp pair p of the CTA shares one shared-memory slot;
// warp half h of the pair holds vectors [h·nvh, h·nvh + nvh) of the row (nvh =
// nv/2, NVH a lane), both shift by the row's first element, and the pair's sums
// meet in shared memory behind the pair's own mbarrier (one arrival per warp,
// a bounded wait), after which half 0's lane 0 refills the slot (both halves
// have copied the row out by then).  With half the registers a warp, a CTA
// holds 24 warps where the one-warp-per-row kernel holds 16, for 12 rows in
// flight: 18.2 against 20.5 µs at h = 6144 (4096 rows), the extra warps hiding
// the arithmetic's latency; at h = 8192, 16 warps (8 rows) where the one-warp
// form holds 8: 27.9 against 28.9 µs back to back.
template <int NVH>
struct LnPairShape {
  static constexpr int MAX_PAIRS = NVH <= 12 ? 12 : 8;  // 24 warps at ≤ 85 registers, or 16 at ≤ 128
};

template <int DT, int NVH>
__global__ void __launch_bounds__(64 * LnPairShape<NVH>::MAX_PAIRS, 1)
    ln_fwd_pair_kernel(ChunkSet cs, const void* __restrict__ gamma, const void* __restrict__ beta, float eps,
                       float* __restrict__ mean, float* __restrict__ rstd, int64_t M, int64_t h, int64_t rpc,
                       unsigned* status, uint64_t timeout_ns) {
  using T = typename Storage<DT>::T;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[LnPairShape<NVH>::MAX_PAIRS];
  __shared__ __align__(8) uint64_t pairbar[LnPairShape<NVH>::MAX_PAIRS];  // one arrival per warp of the pair
  __shared__ float2 xs[LnPairShape<NVH>::MAX_PAIRS][2][2];  // [pair][k & 1][half]
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int pw = w >> 1, half = w & 1;
  const int ppc = blockDim.x >> 6;
  const int nv = static_cast<int>(h / 8);
  const int nvh = nv / 2;
  const uint32_t rb = static_cast<uint32_t>(h * sizeof(T));
  uint4* gs = reinterpret_cast<uint4*>(smem);
  uint4* bs = reinterpret_cast<uint4*>(smem + pad128(rb));
  uint8_t* slot = smem + 2 * pad128(rb) + static_cast<size_t>(pw) * pad128(rb);
  const uint32_t bar = smem_u32(&full[pw]);
  const uint32_t pbar = smem_u32(&pairbar[pw]);
  const int64_t W = static_cast<int64_t>(gridDim.x) * ppc;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * ppc + pw;
  const int64_t cnt = g < M ? (M - g + W - 1) / W : 0;
  const RowStep step(W, rpc);
  RowPos cur(g, step);
  const bool issuer = half == 0 && lane == 0;
  auto issue = [&](const RowPos& at) {
    mbar_arrive_expect_tx(bar, rb);
    bulk_g2s(smem_u32(slot), static_cast<const uint8_t*>(cs.in[at.j]) + at.r * h * static_cast<int64_t>(sizeof(T)),
             rb, bar);
  };
  if (issuer) {
    mbar_init(bar, 1);
    mbar_init(pbar, 2);
    fence_barrier_init();
    if (cnt > 0) issue(cur);
  }
  for (int vi = threadIdx.x; vi < nv; vi += blockDim.x) {
    gs[vi] = __ldg(static_cast<const uint4*>(gamma) + vi);
    bs[vi] = __ldg(static_cast<const uint4*>(beta) + vi);
  }
  __syncthreads();
  const float inv_h = 1.0f / static_cast<float>(h);
  const int v0 = half * nvh;
  for (int64_t k = 0; k < cnt; ++k) {
    const bool ok = mbar_wait_bounded(bar, static_cast<uint32_t>(k & 1), nullptr, status, timeout_ns);
    // (both warps of the pair wait the same bounded time; a give-up is the pair's)
    if (!__all_sync(0xffffffffu, ok)) {
      if (issuer) (void)mbar_wait_bounded(bar, static_cast<uint32_t>(k & 1), nullptr, nullptr, timeout_ns);
      return;
    }
    uint4 v[NVH];
    const uint4* row = reinterpret_cast<const uint4*>(slot);
#pragma unroll
    for (int kk = 0; kk < NVH; ++kk) {
      const int vi = v0 + lane + 32 * kk;
      v[kk] = (lane + 32 * kk < nvh) ? row[vi] : make_uint4(0u, 0u, 0u, 0u);
    }
    float c;  // the row's first element, the same shift for both halves
    {
      float2 f0[4];
      unpack8_pairs<DT>(row[0], f0);
      c = f0[0].x;
    }
    const float2 nc2 = make_float2(-c, -c);
    float2 s1[2], s2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) s1[i] = s2[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int kk = 0; kk < NVH; ++kk) {
      if (lane + 32 * kk < nvh) {
        float2 f[4];
        unpack8_pairs<DT>(v[kk], f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 d = __fadd2_rn(f[i], nc2);
          s1[i & 1] = __fadd2_rn(s1[i & 1], d);
          s2[i & 1] = __ffma2_rn(d, d, s2[i & 1]);
        }
      }
    }
    const float2 t1 = __fadd2_rn(s1[0], s1[1]);
    const float2 t2 = __fadd2_rn(s2[0], s2[1]);
    float q1 = t1.x + t1.y, q2 = t2.x + t2.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      q1 += __shfl_xor_sync(0xffffffffu, q1, o);
      q2 += __shfl_xor_sync(0xffffffffu, q2, o);
    }
    if (lane == 0) xs[pw][k & 1][half] = make_float2(q1, q2);
    __syncwarp();  // this warp's copy out of the slot and its sums are done
    if (lane == 0) mbar_arrive(pbar);
    // the pair's barrier, bounded: a warp that gives up returns, and so does its partner
    const bool pok = mbar_wait_bounded(pbar, static_cast<uint32_t>(k & 1), nullptr, status, timeout_ns);
    if (!__all_sync(0xffffffffu, pok)) return;
    // both halves have copied the row out of the slot: refill it
    if (issuer && k + 1 < cnt) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      RowPos at = cur;
      at.next(step);
      issue(at);
    }
    const float2 a0 = xs[pw][k & 1][0], a1 = xs[pw][k & 1][1];
    const float dm = (a0.x + a1.x) * inv_h;
    const float var = fmaxf((a0.y + a1.y) * inv_h - dm * dm, 0.0f);
    const float mu = c + dm;
    const float r = 1.0f / sqrtf(var + eps);
    reg_fence(v);
    const float2 r2 = make_float2(r, r);
    const float2 nmr2 = make_float2(-mu * r, -mu * r);
    const int64_t m = g + k * W;
    uint4* y = reinterpret_cast<uint4*>(static_cast<T*>(cs.out[cur.j]) + cur.r * h);
#pragma unroll
    for (int kk = 0; kk < NVH; ++kk) {
      if (lane + 32 * kk < nvh) {
        const int vi = v0 + lane + 32 * kk;
        float2 f[4], xh[4];
        unpack8_pairs<DT>(v[kk], f);
#pragma unroll
        for (int i = 0; i < 4; ++i) xh[i] = __ffma2_rn(f[i], r2, nmr2);
        y[vi] = affine8_packed<DT>(pack8_pairs<DT>(xh), lds_v4(gs + vi), lds_v4(bs + vi));
      }
    }
    if (issuer) {
      mean[m] = mu;
      rstd[m] = r;
    }
    cur.next(step);
  }
}

template <int DT, int NVH>
bool ln_fwd_pair_nv(const ChunkSet& cs, const void* gamma, const void* beta, float eps, float* mean, float* rstd,
                    int64_t M, int64_t h, int64_t rpc, cudaStream_t st) {
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != TPMLP_OK || dev == nullptr) return false;
  const size_t slot = pad128(static_cast<uint32_t>(h * 2));
  const size_t fixed = 2 * slot;
  const size_t cap = dev->max_smem_optin > 1024 ? dev->max_smem_optin - 1024 : 0;
  if (cap <= fixed) return false;
  const int ppc = static_cast<int>(std::min<size_t>(LnPairShape<NVH>::MAX_PAIRS, (cap - fixed) / slot));
  if (ppc < 1) return false;
  const size_t smem = fixed + static_cast<size_t>(ppc) * slot;
  auto* fn = ln_fwd_pair_kernel<DT, NVH>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(dev->num_sms, (M + ppc - 1) / ppc)));
  fn<<<grid, 64 * ppc, smem, st>>>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, dev->status, wait_timeout_ns());
  return true;
}

template <int DT, int NV>
bool ln_fwd_warp_nv(const ChunkSet& cs, const void* gamma, const void* beta, float eps, float* mean, float* rstd,
                    int64_t M, int64_t h, int64_t rpc, cudaStream_t st) {
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != TPMLP_OK || dev == nullptr) return false;
  const size_t slot = pad128(static_cast<uint32_t>(h * 2));
  const size_t fixed = 2 * slot;  // γ and β
  const size_t cap = dev->max_smem_optin > 1024 ? dev->max_smem_optin - 1024 : 0;  // static shared memory
  if (cap <= fixed) return false;
  const int wpc = static_cast<int>(std::min<size_t>(LnFwdShape<NV>::MAX_WARPS, (cap - fixed) / slot));
  if (wpc < 1) return false;
  const size_t smem = fixed + static_cast<size_t>(wpc) * slot;
  // (a variant without the per-vector predicate for h = 256·NV held more
  // registers and spilled)
  auto* fn = ln_fwd_warp_kernel<DT, NV, false>;
  // (always set: the kernel's static shared memory counts against the default 48 KB too)
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  // one CTA per SM, and no more warps than rows
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(dev->num_sms, (M + wpc - 1) / wpc)));
  fn<<<grid, 32 * wpc, smem, st>>>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, dev->status, wait_timeout_ns());
  return true;
}

template <int DT>
bool ln_fwd_registers(const ChunkSet& cs, const void* gamma, const void* beta, float eps, float* mean, float* rstd,
                      int64_t M, int64_t h, int64_t rpc, cudaStream_t st) {
  const int64_t per_lane = (h / 8 + 31) / 32;
  if (per_lane <= 4) return ln_fwd_warp_nv<DT, 4>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
  if (per_lane <= 8) return ln_fwd_warp_nv<DT, 8>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
  if (per_lane <= 12) return ln_fwd_warp_nv<DT, 12>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
  if ((h / 8) % 2 == 0 && per_lane > 8 && per_lane <= 24) {
    const int64_t half_lane = (h / 16 + 31) / 32;
    if (half_lane <= 8) return ln_fwd_pair_nv<DT, 8>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
    return ln_fwd_pair_nv<DT, 12>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
  }
  if (per_lane <= 16) return ln_fwd_warp_nv<DT, 16>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
  if (per_lane <= 24) return ln_fwd_warp_nv<DT, 24>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
  if ((h / 8) % 2 == 0 && (h / 16 + 31) / 32 <= 16)
    return ln_fwd_pair_nv<DT, 16>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
  if (per_lane <= REG_MAX_NV) return ln_fwd_warp_nv<DT, 32>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
  return false;
}

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
  const RowStep step(G, rpc);
  RowPos cur(blockIdx.x, step), nxt = cur;  // the row computed, and (thread 0) the next row to load
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_barrier_init();
    for (int64_t k = 0; k < S && k < cnt; ++k) {
      ring_issue(ring, full, cs, static_cast<int>(k), nxt, h, sizeof(T));
      nxt.next(step);
    }
  }
  const float inv_h = 1.0f / static_cast<float>(h);
  int s = 0, s_prev = S - 1;  // slots of rows k and k − 1
  uint32_t ph = 0;            // phase parity of row k's slot
  for (int64_t k = 0; k < cnt; ++k) {
    if (tid == 0 && !mbar_wait_bounded(smem_u32(&full[s]), ph, nullptr, status, timeout_ns)) abort_flag = 1;
    __syncthreads();  // row k is in slot s; every thread is done with row k - 1
    if (abort_flag) {
      if (tid == 0) ring_drain(ring, full, k, cnt, status, timeout_ns);
      return;
    }
    if (tid == 0 && k >= 1 && k - 1 + S < cnt) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ring_issue(ring, full, cs, s_prev, nxt, h, sizeof(T));
      nxt.next(step);
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
    T* y = static_cast<T*>(cs.out[cur.j]) + cur.r * h;
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
    cur.next(step);
    s_prev = s;
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
}

// dx = rstd·(g − mean(g) − x̂·mean(g·x̂)), g = dy·γ, written or added to dx; and
// this CTA's partial sums of dγ = Σ dy·x̂ and dβ = Σ dy over its rows, in row
// order, stored as part[blockIdx.x][:] and part[G + blockIdx.x][:].
// Shared memory: a ring of S slots of (x, dy[, dx being accumulated into])
// rows; thread 0 keeps S − 1 rows in flight while one is computed.  Each thread
// keeps its vectors of γ in registers for the whole kernel and, per row, its
// vectors of x and dy (copied out of the slot once); the dx it accumulates into
// is read from the slot in the second pass; the element-wise math runs on float
// pairs.
template <int DT>
__device__ __forceinline__ void raw_to_pairs(const uint4* raw, float2* f) {
  if constexpr (DT == DT_F32) {
    f[0] = make_float2(__uint_as_float(raw[0].x), __uint_as_float(raw[0].y));
    f[1] = make_float2(__uint_as_float(raw[0].z), __uint_as_float(raw[0].w));
    f[2] = make_float2(__uint_as_float(raw[1].x), __uint_as_float(raw[1].y));
    f[3] = make_float2(__uint_as_float(raw[1].z), __uint_as_float(raw[1].w));
  } else {
    unpack8_pairs_v<DT>(raw[0], f);
  }
}
template <int DT>
__device__ __forceinline__ void pairs_to_raw(const float2* f, uint4* raw) {
  if constexpr (DT == DT_F32) {
    raw[0] = make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x),
                        __float_as_uint(f[1].y));
    raw[1] = make_uint4(__float_as_uint(f[2].x), __float_as_uint(f[2].y), __float_as_uint(f[3].x),
                        __float_as_uint(f[3].y));
  } else {
    raw[0] = pack8_pairs<DT>(f);
  }
}

template <int DT, int V, int THREADS>
__global__ void __launch_bounds__(THREADS, (THREADS == 256 ? 2 : 1)) ln_bwd_stream_kernel(ChunkSet cs, const void* __restrict__ gamma,
                                                                       const float* __restrict__ mean,
                                                                       const float* __restrict__ rstd, int accumulate,
                                                                       float* __restrict__ part, int64_t M, int64_t h,
                                                                       int64_t rpc, int S, unsigned* status,
                                                                       uint64_t timeout_ns) {
  using T = typename Storage<DT>::T;
  constexpr int RAW = DT == DT_F32 ? 2 : 1;  // 16-byte units of an 8-element vector
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[STREAM_MAX_SLOTS];
  __shared__ float2 red[THREADS / 32];
  __shared__ int abort_flag;
  const int tid = threadIdx.x;
  const int nv = static_cast<int>(h / 8);
  const uint32_t rb = static_cast<uint32_t>(h * sizeof(T));
  const RowRing ring{smem, rb, pad128(rb), accumulate ? 3 : 2, S};
  const int64_t G = gridDim.x;
  const int64_t cnt = (M - blockIdx.x + G - 1) / G;
  uint4 graw[V][RAW];  // this thread's vectors of γ
#pragma unroll
  for (int kk = 0; kk < V; ++kk) {
    const int vi = tid + kk * THREADS;
#pragma unroll
    for (int u = 0; u < RAW; ++u)
      graw[kk][u] = vi < nv ? __ldg(reinterpret_cast<const uint4*>(gamma) + vi * RAW + u) : make_uint4(0, 0, 0, 0);
  }
  const RowStep step(G, rpc);
  RowPos cur(blockIdx.x, step), nxt = cur;  // the row computed, and (thread 0) the next row to load
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_barrier_init();
    for (int64_t k = 0; k < S && k < cnt; ++k) {
      ring_issue(ring, full, cs, static_cast<int>(k), nxt, h, sizeof(T));
      nxt.next(step);
    }
  }
  float2 ag[V][4], ab[V][4];
#pragma unroll
  for (int kk = 0; kk < V; ++kk)
#pragma unroll
    for (int i = 0; i < 4; ++i) ag[kk][i] = ab[kk][i] = make_float2(0.0f, 0.0f);
  const float inv_h = 1.0f / static_cast<float>(h);
  float mu_next = cnt > 0 ? mean[blockIdx.x] : 0.0f;
  float r_next = cnt > 0 ? rstd[blockIdx.x] : 0.0f;
  int s = 0, s_prev = S - 1;  // slots of rows k and k − 1
  uint32_t ph = 0;            // phase parity of row k's slot
  for (int64_t k = 0; k < cnt; ++k) {
    const int64_t m = blockIdx.x + k * G;
    const float mu = mu_next, r = r_next;
    if (k + 1 < cnt) {  // the next row's statistics, one row ahead
      mu_next = mean[m + G];
      r_next = rstd[m + G];
    }
    uint4* dx = reinterpret_cast<uint4*>(static_cast<T*>(cs.out[cur.j]) + cur.r * h);
    if (tid == 0 && !mbar_wait_bounded(smem_u32(&full[s]), ph, nullptr, status, timeout_ns)) abort_flag = 1;
    __syncthreads();  // row k is in slot s; every thread is done with row k − 1
    if (abort_flag) {
      if (tid == 0) ring_drain(ring, full, k, cnt, status, timeout_ns);
      return;
    }
    const uint8_t* xs = ring.base + static_cast<size_t>(s) * ring.nin * ring.rb_al;
    const uint8_t* ds = xs + ring.rb_al;
    const uint8_t* os = xs + 2 * ring.rb_al;  // the dx being accumulated into (accumulate only)
    uint4 xraw[V][RAW], draw[V][RAW];
#pragma unroll
    for (int kk = 0; kk < V; ++kk) {
      const int vi = tid + kk * THREADS;
#pragma unroll
      for (int u = 0; u < RAW; ++u) {
        xraw[kk][u] = vi < nv ? reinterpret_cast<const uint4*>(xs)[vi * RAW + u] : make_uint4(0, 0, 0, 0);
        draw[kk][u] = vi < nv ? reinterpret_cast<const uint4*>(ds)[vi * RAW + u] : make_uint4(0, 0, 0, 0);
      }
    }
    if (tid == 0 && k >= 1 && k - 1 + S < cnt) {  // row k − 1's slot is free
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ring_issue(ring, full, cs, s_prev, nxt, h, sizeof(T));
      nxt.next(step);
    }
    const float2 r2 = make_float2(r, r), nmr2 = make_float2(-mu * r, -mu * r);
    float2 sg1 = make_float2(0.0f, 0.0f), sgx = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int kk = 0; kk < V; ++kk) {
      if (tid + kk * THREADS < nv) {
        float2 xv[4], d[4], g[4];
        raw_to_pairs<DT>(xraw[kk], xv);
        raw_to_pairs<DT>(draw[kk], d);
        raw_to_pairs<DT>(graw[kk], g);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 xh = __ffma2_rn(xv[i], r2, nmr2);
          const float2 gi = __fmul2_rn(d[i], g[i]);
          sg1 = __fadd2_rn(sg1, gi);
          sgx = __ffma2_rn(gi, xh, sgx);
          ag[kk][i] = __ffma2_rn(d[i], xh, ag[kk][i]);
          ab[kk][i] = __fadd2_rn(ab[kk][i], d[i]);
        }
      }
    }
    // red[] is free: every thread passed this row's first barrier after its last read
    const float2 tot = block_sum2_free<THREADS>(sg1.x + sg1.y, sgx.x + sgx.y, red);
    const float2 nmg2 = make_float2(-tot.x * inv_h, -tot.x * inv_h);
    const float2 nmgx2 = make_float2(-tot.y * inv_h, -tot.y * inv_h);
#pragma unroll
    for (int kk = 0; kk < V; ++kk) {
      const int vi = tid + kk * THREADS;
      if (vi < nv) {
        float2 xv[4], d[4], g[4], o[4];
        raw_to_pairs<DT>(xraw[kk], xv);
        raw_to_pairs<DT>(draw[kk], d);
        raw_to_pairs<DT>(graw[kk], g);
        if (accumulate) {
          uint4 oraw[RAW];
#pragma unroll
          for (int u = 0; u < RAW; ++u) oraw[u] = reinterpret_cast<const uint4*>(os)[vi * RAW + u];
          raw_to_pairs<DT>(oraw, o);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 xh = __ffma2_rn(xv[i], r2, nmr2);
          const float2 t = __ffma2_rn(xh, nmgx2, __ffma2_rn(d[i], g[i], nmg2));  // g − mean(g) − x̂·mean(g·x̂)
          o[i] = accumulate ? __ffma2_rn(t, r2, o[i]) : __fmul2_rn(t, r2);
        }
        uint4 out[RAW];
        pairs_to_raw<DT>(o, out);
#pragma unroll
        for (int u = 0; u < RAW; ++u) dx[vi * RAW + u] = out[u];
      }
    }
    cur.next(step);
    s_prev = s;
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
  float* pg = part + static_cast<int64_t>(blockIdx.x) * h;
  float* pb = part + (G + blockIdx.x) * h;
#pragma unroll
  for (int kk = 0; kk < V; ++kk) {
    const int vi = tid + kk * THREADS;
    if (vi < nv) {
      float4* qg = reinterpret_cast<float4*>(pg + static_cast<int64_t>(vi) * 8);
      float4* qb = reinterpret_cast<float4*>(pb + static_cast<int64_t>(vi) * 8);
      qg[0] = make_float4(ag[kk][0].x, ag[kk][0].y, ag[kk][1].x, ag[kk][1].y);
      qg[1] = make_float4(ag[kk][2].x, ag[kk][2].y, ag[kk][3].x, ag[kk][3].y);
      qb[0] = make_float4(ab[kk][0].x, ab[kk][0].y, ab[kk][1].x, ab[kk][1].y);
      qb[1] = make_float4(ab[kk][2].x, ab[kk][2].y, ab[kk][3].x, ab[kk][3].y);
    }
  }
}

// dγ[c], dβ[c] from the G per-CTA partials (part = [dγ rows G | dβ rows G] of h,
// h a multiple of 4): a CTA takes 64 consecutive columns of [dγ | dβ] as 16
// float4 quads, its 32 row groups add the rows g ≡ group (mod 32) with every
// load independent of the others, and the 32 group sums are added in group
// order — the same association on every run.
constexpr int RP_QUADS = 16, RP_GROUPS = 32;

__global__ void __launch_bounds__(RP_QUADS * RP_GROUPS) ln_bwd_reduce_parts_kernel(const float* __restrict__ part,
                                                                                   float* __restrict__ dgamma,
                                                                                   float* __restrict__ dbeta,
                                                                                   int64_t h, int64_t G) {
  __shared__ float4 acc[RP_GROUPS][RP_QUADS];
  const int tx = threadIdx.x % RP_QUADS, ty = threadIdx.x / RP_QUADS;
  const int64_t col = (static_cast<int64_t>(blockIdx.x) * RP_QUADS + tx) * 4;  // over [dγ | dβ], 2h columns
  float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (col < 2 * h) {
    const int64_t which = col >= h ? 1 : 0;
    const float4* p = reinterpret_cast<const float4*>(part + which * G * h + (col - which * h));
    const int64_t step = h / 4;  // float4s per partial row
#pragma unroll 8
    for (int64_t g = ty; g < G; g += RP_GROUPS) {
      const float4 v = __ldcs(p + g * step);
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
  }
  acc[ty][tx] = a;
  __syncthreads();
  if (ty == 0 && col < 2 * h) {
    float4 t = acc[0][tx];
#pragma unroll
    for (int y = 1; y < RP_GROUPS; ++y) {
      const float4 u = acc[y][tx];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    float* out = col < h ? dgamma + col : dbeta + (col - h);  // 4-byte aligned: scalar stores
    out[0] = t.x;
    out[1] = t.y;
    out[2] = t.z;
    out[3] = t.w;
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

StreamPlan plan_stream(const void* fn, size_t fixed, size_t slot, int ctas_per_sm, int64_t max_grid,
                       int threads = STREAM_THREADS) {
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
  // (always set: the kernel's static shared memory counts against the default 48 KB too)
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return p;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, smem) != cudaSuccess || occ < 1) {
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

template <int DT, int V, int THREADS>
bool ln_bwd_streamed_v(const ChunkSet& cs, const void* gamma, const float* mean, const float* rstd, int accumulate,
                       float* dgamma, float* dbeta, float* part, int64_t max_parts, int64_t M, int64_t h, int64_t rpc,
                       cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(ln_bwd_stream_kernel<DT, V, THREADS>);
  const size_t rb = pad128(static_cast<uint32_t>(h * sizeof(typename Storage<DT>::T)));
  const StreamPlan p = plan_stream(fn, 0, (accumulate ? 3 : 2) * rb, THREADS == 256 ? 2 : 1, std::min(M, max_parts),
                                   THREADS);
  if (!p.ok) return false;
  DeviceInfo* dev = nullptr;
  current_device(&dev);
  ln_bwd_stream_kernel<DT, V, THREADS><<<p.grid, THREADS, p.smem, st>>>(cs, gamma, mean, rstd, accumulate, part, M, h,
                                                                       rpc, p.S, dev->status, wait_timeout_ns());
  ln_bwd_reduce_parts_kernel<<<static_cast<unsigned>((2 * h / 4 + RP_QUADS - 1) / RP_QUADS), RP_QUADS * RP_GROUPS, 0,
                               st>>>(part, dgamma, dbeta, h, p.grid);
  return true;
}

// Threads per CTA and vectors per thread for a row of nv 8-element vectors:
// 256 threads and two CTAs per SM (so that one CTA's barrier waits are covered
// by the other's work) up to three vectors a thread; wider rows, 512 threads.
template <int DT>
bool ln_bwd_streamed(const ChunkSet& cs, const void* gamma, const float* mean, const float* rstd, int accumulate,
                     float* dgamma, float* dbeta, float* part, int64_t max_parts, int64_t M, int64_t h, int64_t rpc,
                     cudaStream_t st) {
  const int64_t nv = h / 8;
#define LNBS(V, TH) \
  return ln_bwd_streamed_v<DT, V, TH>(cs, gamma, mean, rstd, accumulate, dgamma, dbeta, part, max_parts, M, h, rpc, st)
  if (nv <= 256) LNBS(1, 256);
  if (nv <= 512) LNBS(2, 256);
  if (nv <= 768) LNBS(3, 256);
  if (nv <= 1024) LNBS(2, 512);
#undef LNBS
  return false;
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
  if (vec && dtype != DT_F32) {
    // 16-bit rows up to h = 8192: a warp per row, the row in registers
    streamed = dtype == DT_F16 ? ln_fwd_registers<DT_F16>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st)
                               : ln_fwd_registers<DT_BF16>(cs, gamma, beta, eps, mean, rstd, M, h, rpc, st);
  }
  if (!streamed && vec && h >= STREAM_MIN_H && h <= 8 * STREAM_THREADS * STREAM_MAX_V) {
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
