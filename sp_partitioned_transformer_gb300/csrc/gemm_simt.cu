// Float32 GEMM on the CUDA cores for the float32 storage type.
//
// The tensor cores have no float32 path that keeps a 1e-5 relative error
// (TF32 rounds the inputs to 10 mantissa bits), so the float32 block runs the
// same contractions and epilogues as the tensor-core kernel, here as a plain
// shared-memory tiled GEMM: 64×64 output tile per CTA, 16-deep K slices, 4×4
// outputs per thread, any shape, any operand majorness, any alignment.  The
// accumulator tile is staged through shared memory so that the SwiGLU epilogue
// can pair each gate column with its up column.
#include <algorithm>

#include "internal.h"

namespace tpmlp {
namespace simt {

constexpr int TM = 64, TN = 64, TK = 16, THREADS = 256;
constexpr int MAX_SEGS = 16, MAX_PARTS = 16;

struct Params {
  const float* a[MAX_SEGS];
  const float* b[MAX_SEGS];
  int64_t k[MAX_SEGS];
  int32_t seg_begin[MAX_PARTS + 1];
  int32_t a_mn, b_mn;
  int64_t lda, ldb;
  int64_t M, N;
  int64_t swiglu_up_row;
  int32_t part_base;
  int32_t pad;
  EpiParams epi;
};

__device__ __forceinline__ void epi_scalar(const Params& p, int64_t m, int64_t n, float v, int part) {
  const EpiParams& e = p.epi;
  switch (e.kind) {
    case EPI_F32:
      static_cast<float*>(e.out)[static_cast<int64_t>(part) * e.part_stride + m * e.ldo + n] = v;
      return;
    case EPI_ACC_F32:
      static_cast<float*>(e.out)[m * e.ldo + n] += v;
      return;
    case EPI_STORE: {
      float* row;
      if (e.scatter) {
        const int64_t sh = m / e.rows_per_shard;
        row = static_cast<float*>(e.shard[sh]) + (m - sh * e.rows_per_shard) * e.ldo;
      } else {
        row = static_cast<float*>(e.out) + m * e.ldo;
      }
      row[n] = v;
      return;
    }
    case EPI_ACT:
      static_cast<float*>(e.out)[m * e.ldo + n] = v;
      static_cast<float*>(e.out2)[m * e.ldo2 + n] = act_fwd<true>(e.act, v);
      return;
    default: {  // EPI_DACT
      const float* u = static_cast<const float*>(e.aux) + m * e.ldaux;
      float* du = static_cast<float*>(e.out) + m * e.ldo;
      if (e.act == ACT_SWIGLU) {
        const float g = u[n], up = u[e.swiglu_F + n];
        const float s = sigmoid_f<true>(g);
        du[n] = v * up * (s * (1.0f + g * (1.0f - s)));
        du[e.swiglu_F + n] = v * (g * s);
      } else {
        du[n] = v * act_grad<true>(e.act, u[n]);
      }
      return;
    }
  }
}

__global__ void __launch_bounds__(THREADS) gemm_kernel(const __grid_constant__ Params p) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  __shared__ float Cs[TM][TN + 1];
  const int part = blockIdx.z;
  const bool swiglu = p.swiglu_up_row > 0;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * (swiglu ? TN / 2 : TN);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int si = p.seg_begin[part]; si < p.seg_begin[part + 1]; ++si) {
    const float* A = p.a[si];
    const float* B = p.b[si];
    const int64_t K = p.k[si];
    for (int64_t k0 = 0; k0 < K; k0 += TK) {
      for (int i = threadIdx.x; i < TM * TK; i += THREADS) {
        // coalesce along the operand's contiguous dimension
        const int mm = p.a_mn ? i % TM : i / TK;
        const int kk = p.a_mn ? i / TM : i % TK;
        const int64_t gm = m0 + mm, gk = k0 + kk;
        float v = 0.0f;
        if (gm < p.M && gk < K) v = p.a_mn ? A[gk * p.lda + gm] : A[gm * p.lda + gk];
        As[kk][mm] = v;
      }
      for (int i = threadIdx.x; i < TN * TK; i += THREADS) {
        const int nn = p.b_mn ? i % TN : i / TK;
        const int kk = p.b_mn ? i / TN : i % TK;
        int64_t logical, brow;
        if (swiglu) {
          logical = n0 + (nn % (TN / 2));
          brow = nn < TN / 2 ? logical : p.swiglu_up_row + logical;
        } else {
          logical = n0 + nn;
          brow = logical;
        }
        const int64_t gk = k0 + kk;
        float v = 0.0f;
        if (logical < p.N && gk < K) v = p.b_mn ? B[gk * p.ldb + brow] : B[brow * p.ldb + gk];
        Bs[kk][nn] = v;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < TK; ++kk) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) Cs[ty * 4 + i][tx * 4 + j] = acc[i][j];
  __syncthreads();

  const EpiParams& e = p.epi;
  for (int i = threadIdx.x; i < TM * TN; i += THREADS) {
    const int r = i / TN, c = i % TN;
    const int64_t m = m0 + r;
    if (m >= p.M) continue;
    if (swiglu) {
      if (c >= TN / 2) continue;
      const int64_t n = n0 + c;
      if (n >= p.N) continue;
      const float g = Cs[r][c], up = Cs[r][c + TN / 2];
      static_cast<float*>(e.out)[m * e.ldo + n] = g;
      static_cast<float*>(e.out)[m * e.ldo + e.swiglu_F + n] = up;
      static_cast<float*>(e.out2)[m * e.ldo2 + n] = g * sigmoid_f<true>(g) * up;
    } else {
      const int64_t n = n0 + c;
      if (n >= p.N) continue;
      epi_scalar(p, m, n, Cs[r][c], p.part_base + part);
    }
  }
}

}  // namespace simt

int launch_gemm_simt(const GemmDesc& g, cudaStream_t st) {
  using namespace simt;
  if (g.M <= 0 || g.N <= 0) return TPMLP_OK;
  Params p;
  memset(&p, 0, sizeof(p));
  p.a_mn = g.a_mn;
  p.b_mn = g.b_mn;
  p.lda = g.lda;
  p.ldb = g.ldb;
  p.M = g.M;
  p.N = g.N;
  p.swiglu_up_row = g.swiglu_up_row;
  p.epi = g.epi;
  const int64_t tile_n = g.swiglu_up_row > 0 ? TN / 2 : TN;
  const int nseg = static_cast<int>(g.segs.size());
  int seg_i = 0, part = 0;
  while (part < g.nparts) {
    int nparts = 0, nsegs = 0;
    p.part_base = part;
    p.seg_begin[0] = 0;
    while (part < g.nparts && nparts < MAX_PARTS) {
      int cnt = 0;
      while (seg_i + nsegs + cnt < nseg && g.segs[seg_i + nsegs + cnt].part == part) ++cnt;
      if (cnt == 0) return set_error(TPMLP_ERR_INVALID_ARG, "a GEMM partial has no K segment");
      if (nsegs + cnt > MAX_SEGS) {
        if (nparts == 0) return set_error(TPMLP_ERR_UNSUPPORTED, "too many K segments in one partial");
        break;
      }
      for (int c = 0; c < cnt; ++c) {
        const GemmSeg& s = g.segs[seg_i + nsegs + c];
        p.a[nsegs + c] = static_cast<const float*>(s.a);
        p.b[nsegs + c] = static_cast<const float*>(s.b);
        p.k[nsegs + c] = s.k;
      }
      nsegs += cnt;
      ++nparts;
      p.seg_begin[nparts] = nsegs;
      ++part;
    }
    const int64_t gx = (g.N + tile_n - 1) / tile_n, gy = (g.M + TM - 1) / TM;
    if (gx >= (1ll << 31) || gy > 65535) return set_error(TPMLP_ERR_UNSUPPORTED, "float32 GEMM grid too large");
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(nparts));
    double ksum = 0.0;
    for (int c = 0; c < nsegs; ++c) ksum += static_cast<double>(p.k[c]);
    const int ph = prof_begin(PROF_GEMM_SIMT, st);
    gemm_kernel<<<grid, THREADS, 0, st>>>(p);
    prof_end(ph, 2.0 * static_cast<double>(g.M) * static_cast<double>(g.swiglu_up_row > 0 ? 2 * g.N : g.N) * ksum, st);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("float32 GEMM launch: ") + cudaGetErrorString(e));
    seg_i += nsegs;
  }
  return TPMLP_OK;
}

}  // namespace tpmlp
