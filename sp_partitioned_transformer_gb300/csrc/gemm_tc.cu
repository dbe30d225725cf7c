// Tensor-core GEMM for the six contractions of the MLP block (sm_103a).
//
//   C[m, n] = Σ_segments Σ_k A(m, k)·B(n, k)   (float32 accumulation in TMEM)
//
// covering: fc1 column-parallel forward (U_i = X·A_i, GeLU/SwiGLU epilogue),
// fc2 row-parallel forward (P_i = Y_i·B_i as float32 partials, or the shard sum
// folded into one accumulator), fc2 input gradient with the activation
// derivative fused (dU_i = act'(U_i) ⊙ dZ·B_iᵀ), both weight gradients
// (dB_i = Y_iᵀ·dZ, dA_i = Xᵀ·dU_i) and fc1's input gradient (Σ_i dU_i·A_iᵀ)
// ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §2–§5;
// "tensor-parallelism-matrix-split", §Backward：为什么有些梯度需要求和).
//
// Design (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: 128-byte-swizzled 128×64 A and 256×64 B tiles
//               into a 4-stage shared-memory ring (mbarrier full/empty pairs);
//   warp 1      MMA issuer: tcgen05.mma cta_group::1 M=128 N=256 K=16 from
//               shared-memory descriptors into one of two TMEM accumulators;
//   warp 2      TMEM allocator (512 columns = two 128×256 fp32 accumulators);
//   warps 4-7   epilogue: tcgen05.ld of the finished accumulator (each warp its
//               32-lane quarter), activation math, 16-byte global stores, so the
//               epilogue of tile t overlaps the MMAs of tile t+1.
// K-major and MN-major operands are both read straight from their row-major
// storage: for MN-major operands TMA loads 64(MN)×64(K) boxes and the UMMA
// descriptor walks them with LBO = 8 KB (next 64-wide MN block) and SBO = 1 KB
// (next 8 K-rows).  Ragged M, N and K are covered by TMA's zero fill and
// predicated stores.  Every mbarrier wait is bounded (device status word).
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "internal.h"

namespace tpmlp {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // 64 16-bit elements = one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int THREADS = 256;
constexpr int MAX_MAPS = 32;
constexpr int MAX_SEGS = 16;
constexpr int MAX_PARTS = 16;
constexpr int GROUP_M = 16;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr size_t SMEM_BYTES = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + 256;

// MN-major box: 64 elements along M/N (128 bytes) × 64 K-rows = 8 KB.
constexpr uint32_t MN_BOX_BYTES = 64 * BK * 2;

struct Seg {
  int32_t map_a, map_b, k_len, pad;
};

struct Params {
  CUtensorMap maps[MAX_MAPS];
  Seg segs[MAX_SEGS];
  int32_t seg_begin[MAX_PARTS + 1];
  int32_t M, N;           // logical output extent (N = F for SwiGLU fc1)
  int32_t mt, nt;         // tile counts along M and N
  int32_t nparts;         // output partials handled by this launch
  int32_t part_base;      // index of this launch's first partial
  int32_t swiglu_up_row;  // > 0: SwiGLU fc1, B rows of the up half start here
  int32_t pad0;
  unsigned* status;
  uint64_t timeout_ns;
  EpiParams epi;
};

__device__ __forceinline__ void decode_tile(int t, const Params& p, int& part, int& mb, int& nb) {
  const int per_part = p.mt * p.nt;
  part = t / per_part;
  const int r = t - part * per_part;
  const int span = GROUP_M * p.nt;
  const int g = r / span;
  const int first_m = g * GROUP_M;
  const int gsz = min(p.mt - first_m, GROUP_M);
  const int rr = r - g * span;
  mb = first_m + rr % gsz;
  nb = rr / gsz;
}

// ---------------------------------------------------------------- epilogues
template <int DT>
__device__ __forceinline__ void epi_chunk(const Params& p, int64_t m, int64_t n0, const float* v,
                                          int part) {
  using T = typename Storage<DT>::T;
  const EpiParams& e = p.epi;
  const int64_t N = p.N;
  if (e.kind == EPI_F32) {
    float* o = static_cast<float*>(e.out) + static_cast<int64_t>(part) * e.part_stride + m * e.ldo + n0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (n0 + 4 * j < N)
        reinterpret_cast<float4*>(o)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    return;
  }
  if (e.kind == EPI_STORE) {
    T* row;
    if (e.scatter) {
      const int64_t sh = m / e.rows_per_shard;
      row = static_cast<T*>(e.shard[sh]) + (m - sh * e.rows_per_shard) * e.ldo;
    } else {
      row = static_cast<T*>(e.out) + m * e.ldo;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (n0 + 8 * j < N) *reinterpret_cast<uint4*>(row + n0 + 8 * j) = pack8<DT>(v + 8 * j);
    return;
  }
  if (e.kind == EPI_ACT) {
    T* u = static_cast<T*>(e.out) + m * e.ldo + n0;
    T* y = static_cast<T*>(e.out2) + m * e.ldo2 + n0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (n0 + 8 * j < N) {
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = act_fwd<false>(e.act, v[8 * j + i]);
        *reinterpret_cast<uint4*>(u + 8 * j) = pack8<DT>(v + 8 * j);
        *reinterpret_cast<uint4*>(y + 8 * j) = pack8<DT>(a);
      }
    }
    return;
  }
  // EPI_DACT
  if (e.act == ACT_SWIGLU) {
    // dY chunk -> dG = dY·Up·silu'(G), dUp = dY·silu(G); G, Up from the saved U.
    const T* ug = static_cast<const T*>(e.aux) + m * e.ldaux + n0;
    const T* uu = ug + e.swiglu_F;
    T* dg = static_cast<T*>(e.out) + m * e.ldo + n0;
    T* du = dg + e.swiglu_F;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (n0 + 8 * j < N) {
        float g[8], up[8], rg[8], ru[8];
        unpack8<DT>(*reinterpret_cast<const uint4*>(ug + 8 * j), g);
        unpack8<DT>(*reinterpret_cast<const uint4*>(uu + 8 * j), up);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float s = sigmoid_f<false>(g[i]);
          const float dy = v[8 * j + i];
          rg[i] = dy * up[i] * (s * (1.0f + g[i] * (1.0f - s)));
          ru[i] = dy * (g[i] * s);
        }
        *reinterpret_cast<uint4*>(dg + 8 * j) = pack8<DT>(rg);
        *reinterpret_cast<uint4*>(du + 8 * j) = pack8<DT>(ru);
      }
    }
    return;
  }
  const T* u = static_cast<const T*>(e.aux) + m * e.ldaux + n0;
  T* du = static_cast<T*>(e.out) + m * e.ldo + n0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (n0 + 8 * j < N) {
      float uf[8], d[8];
      unpack8<DT>(*reinterpret_cast<const uint4*>(u + 8 * j), uf);
#pragma unroll
      for (int i = 0; i < 8; ++i) d[i] = v[8 * j + i] * act_grad<false>(e.act, uf[i]);
      *reinterpret_cast<uint4*>(du + 8 * j) = pack8<DT>(d);
    }
  }
}

// SwiGLU fc1: 32 gate and the matching 32 up columns of one row.
template <int DT>
__device__ __forceinline__ void epi_swiglu_fwd(const Params& p, int64_t m, int64_t n0,
                                               const float* g, const float* up) {
  using T = typename Storage<DT>::T;
  const EpiParams& e = p.epi;
  T* ug = static_cast<T*>(e.out) + m * e.ldo + n0;
  T* uu = ug + e.swiglu_F;
  T* y = static_cast<T*>(e.out2) + m * e.ldo2 + n0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (n0 + 8 * j < p.N) {
      float a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float x = g[8 * j + i];
        a[i] = x * sigmoid_f<false>(x) * up[8 * j + i];
      }
      *reinterpret_cast<uint4*>(ug + 8 * j) = pack8<DT>(g + 8 * j);
      *reinterpret_cast<uint4*>(uu + 8 * j) = pack8<DT>(up + 8 * j);
      *reinterpret_cast<uint4*>(y + 8 * j) = pack8<DT>(a);
    }
  }
}

// ---------------------------------------------------------------- kernel
template <int DT, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(THREADS, 1) gemm_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment of the tile ring (128-byte swizzle atoms are 1 KB).
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + STAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * STAGES);
  const uint32_t tempty0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8u * a, 1);
      mbar_init(tempty0 + 8u * a, 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_tiles = p.mt * p.nt * p.nparts;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int s = p.seg_begin[0]; s < p.seg_begin[p.nparts]; ++s) {
        tma_prefetch_map(&p.maps[p.segs[s].map_a]);
        tma_prefetch_map(&p.maps[p.segs[s].map_b]);
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        int part, mb, nb;
        decode_tile(t, p, part, mb, nb);
        for (int si = p.seg_begin[part]; ok && si < p.seg_begin[part + 1]; ++si) {
          const Seg sg = p.segs[si];
          const CUtensorMap* ma = &p.maps[sg.map_a];
          const CUtensorMap* mbp = &p.maps[sg.map_b];
          const int nkb = (sg.k_len + BK - 1) / BK;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait_bounded(empty0 + 8u * stage, phase ^ 1u, abort_flag, p.status, p.timeout_ns)) {
              ok = false;
              break;
            }
            const uint32_t fb = full0 + 8u * stage;
            mbar_arrive_expect_tx(fb, STAGE_BYTES);
            const uint32_t sa = smem_u32(smem_a + stage * A_BYTES);
            const uint32_t sb = smem_u32(smem_b + stage * B_BYTES);
            const int k0 = kb * BK;
            if constexpr (!A_MN) {
              tma_load_2d(sa, ma, fb, k0, mb * BM);
            } else {
              tma_load_2d(sa, ma, fb, mb * BM, k0);
              tma_load_2d(sa + MN_BOX_BYTES, ma, fb, mb * BM + 64, k0);
            }
            if constexpr (!B_MN) {
              if (p.swiglu_up_row > 0) {
                tma_load_2d(sb, mbp, fb, k0, nb * (BN / 2));
                tma_load_2d(sb + B_BYTES / 2, mbp, fb, k0, p.swiglu_up_row + nb * (BN / 2));
              } else {
                tma_load_2d(sb, mbp, fb, k0, nb * BN);
              }
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + j * MN_BOX_BYTES, mbp, fb, nb * BN + j * 64, k0);
            }
            issued_mask |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        for (int s = 0; s < STAGES; ++s)
          if ((issued_mask >> s) & 1u)
            (void)mbar_wait_bounded(full0 + 8u * s, (issued_phase >> s) & 1u, nullptr, nullptr, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_f16(DT == DT_BF16, A_MN, B_MN, BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x, ++it) {
        int part, mb, nb;
        decode_tile(t, p, part, mb, nb);
        const int acc = it & 1;
        const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
        if (!mbar_wait_bounded(tempty0 + 8u * acc, acc_phase ^ 1u, abort_flag, p.status, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        uint32_t accumulate = 0;
        for (int si = p.seg_begin[part]; ok && si < p.seg_begin[part + 1]; ++si) {
          const int nkb = (p.segs[si].k_len + BK - 1) / BK;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait_bounded(full0 + 8u * stage, phase, abort_flag, p.status, p.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem_a + stage * A_BYTES);
            const uint32_t sb = smem_u32(smem_b + stage * B_BYTES);
#pragma unroll
            for (int ks = 0; ks < BK / UMMA_K; ++ks) {
              // K-major: the next 16 K-elements are 32 bytes further along each
              // swizzled 128-byte row.  MN-major: 16 K-rows = two 1 KB atoms.
              const uint64_t ad = A_MN ? make_sdesc_sw128(sa + ks * 2048u, MN_BOX_BYTES, 1024u)
                                       : make_sdesc_sw128(sa + ks * 32u, 16u, 1024u);
              const uint64_t bd = B_MN ? make_sdesc_sw128(sb + ks * 2048u, MN_BOX_BYTES, 1024u)
                                       : make_sdesc_sw128(sb + ks * 32u, 16u, 1024u);
              tc_mma_f16(d_tmem, ad, bd, idesc, accumulate);
              accumulate = 1u;
            }
            tc_commit(empty0 + 8u * stage);  // frees the stage once these MMAs finish
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        tc_commit(tfull0 + 8u * acc);  // accumulator ready for the epilogue
      }
      if (!ok) {
        tc_commit(drain_bar);
        (void)mbar_wait_bounded(drain_bar, 0u, nullptr, nullptr, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter accessible to this warp
    const bool swiglu_fwd = p.swiglu_up_row > 0;
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      int part, mb, nb;
      decode_tile(t, p, part, mb, nb);
      const int acc = it & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
      const bool ok = mbar_wait_bounded(tfull0 + 8u * acc, acc_phase, abort_flag, p.status, p.timeout_ns);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int64_t m = static_cast<int64_t>(mb) * BM + q * 32 + lane;
      const bool row_ok = m < p.M;
      const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if (swiglu_fwd) {
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          float g[32], up[32];
          tmem_ld32(trow + c * 32, g);
          tmem_ld32(trow + BN / 2 + c * 32, up);
          if (row_ok) epi_swiglu_fwd<DT>(p, m, static_cast<int64_t>(nb) * (BN / 2) + c * 32, g, up);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(trow + c * 32, v);
          if (row_ok) epi_chunk<DT>(p, m, static_cast<int64_t>(nb) * BN + c * 32, v, p.part_base + part);
        }
      }
      tc_fence_before();
      mbar_arrive(tempty0 + 8u * acc);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  });
  return fn;
}

// 2-D map over a row-major [outer, inner] matrix with row pitch ld (elements).
static int make_map(CUtensorMap* m, int dtype, const void* base, int64_t inner, int64_t outer,
                    int64_t ld, uint32_t box_inner, uint32_t box_outer) {
  EncodeFn enc = get_encode();
  if (!enc) return set_error(TPMLP_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(m, dtype == DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(TPMLP_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string(static_cast<int>(r)) + ")");
  return TPMLP_OK;
}

template <int DT, bool A_MN, bool B_MN>
static int launch_one(const Params& p, int grid, cudaStream_t st, const DeviceInfo& dev) {
  static std::mutex mu;
  static bool attr_set[64] = {};
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev.device >= 0 && dev.device < 64 && !attr_set[dev.device]) {
      const cudaError_t e = cudaFuncSetAttribute(gemm_kernel<DT, A_MN, B_MN>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(SMEM_BYTES));
      if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
      attr_set[dev.device] = true;
    }
  }
  gemm_kernel<DT, A_MN, B_MN><<<grid, THREADS, SMEM_BYTES, st>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("tensor-core GEMM launch: ") + cudaGetErrorString(e));
  return TPMLP_OK;
}

template <int DT>
static int dispatch(const Params& p, int grid, cudaStream_t st, const DeviceInfo& dev, bool a_mn, bool b_mn) {
  if (!a_mn && !b_mn) return launch_one<DT, false, false>(p, grid, st, dev);
  if (!a_mn && b_mn) return launch_one<DT, false, true>(p, grid, st, dev);
  if (a_mn && b_mn) return launch_one<DT, true, true>(p, grid, st, dev);
  return set_error(TPMLP_ERR_UNSUPPORTED, "MN-major A with K-major B is not instantiated");
}

}  // namespace tc

int launch_gemm_tc(const GemmDesc& g, cudaStream_t st) {
  using namespace tc;
  DeviceInfo* dev = nullptr;
  int rc = current_device(&dev);
  if (rc != TPMLP_OK) return rc;
  if (g.M <= 0 || g.N <= 0) return TPMLP_OK;
  if (g.M >= (1ll << 31) || g.N >= (1ll << 31)) return set_error(TPMLP_ERR_UNSUPPORTED, "GEMM extent >= 2^31");
  const bool swiglu = g.swiglu_up_row > 0;
  if (swiglu && (g.a_mn || g.b_mn)) return set_error(TPMLP_ERR_UNSUPPORTED, "SwiGLU pairing needs K-major operands");

  Params p;
  memset(&p, 0, sizeof(p));
  p.M = static_cast<int32_t>(g.M);
  p.N = static_cast<int32_t>(g.N);
  p.mt = static_cast<int32_t>((g.M + BM - 1) / BM);
  const int tile_n = swiglu ? BN / 2 : BN;
  p.nt = static_cast<int32_t>((g.N + tile_n - 1) / tile_n);
  p.swiglu_up_row = static_cast<int32_t>(g.swiglu_up_row);
  p.status = dev->status;
  p.timeout_ns = wait_timeout_ns();
  p.epi = g.epi;

  // Launch batches: consecutive partials whose segments fit the parameter block.
  int seg_i = 0;
  const int nseg = static_cast<int>(g.segs.size());
  int part = 0;
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
        if (s.k <= 0 || s.k >= (1ll << 31)) return set_error(TPMLP_ERR_INVALID_ARG, "bad K segment");
        const int idx = nsegs + c;
        Seg& d = p.segs[idx];
        d.map_a = 2 * idx;
        d.map_b = 2 * idx + 1;
        d.k_len = static_cast<int32_t>(s.k);
        if (!g.a_mn)
          rc = make_map(&p.maps[d.map_a], g.dtype, s.a, s.k, g.M, g.lda, BK, BM);
        else
          rc = make_map(&p.maps[d.map_a], g.dtype, s.a, g.M, s.k, g.lda, 64, BK);
        if (rc != TPMLP_OK) return rc;
        if (!g.b_mn)
          rc = make_map(&p.maps[d.map_b], g.dtype, s.b, s.k, g.b_rows, g.ldb, BK, swiglu ? BN / 2 : BN);
        else
          rc = make_map(&p.maps[d.map_b], g.dtype, s.b, g.N, s.k, g.ldb, 64, BK);
        if (rc != TPMLP_OK) return rc;
      }
      nsegs += cnt;
      ++nparts;
      p.seg_begin[nparts] = nsegs;
      ++part;
    }
    p.nparts = nparts;
    const int64_t tiles = static_cast<int64_t>(p.mt) * p.nt * nparts;
    if (tiles >= (1ll << 31)) return set_error(TPMLP_ERR_UNSUPPORTED, "too many tiles");
    const int grid = static_cast<int>(std::min<int64_t>(tiles, dev->num_sms));
    double ksum = 0.0;
    for (int c = 0; c < nsegs; ++c) ksum += static_cast<double>(p.segs[c].k_len);
    const double work = 2.0 * static_cast<double>(g.M) * static_cast<double>(swiglu ? 2 * g.N : g.N) * ksum;
    const int ph = prof_begin(PROF_GEMM_TC, st);
    if (g.dtype == DT_BF16)
      rc = dispatch<DT_BF16>(p, grid, st, *dev, g.a_mn, g.b_mn);
    else
      rc = dispatch<DT_F16>(p, grid, st, *dev, g.a_mn, g.b_mn);
    prof_end(ph, work, st);
    if (rc != TPMLP_OK) return rc;
    seg_i += nsegs;
  }
  return TPMLP_OK;
}

}  // namespace tpmlp
