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
// Two kernels: gemm_pair_kernel (every GEMM with M > 128) computes 256×256
// tiles on CTA pairs (clusters of 2) with tcgen05.mma cta_group::2 and a
// 6-stage ring, each CTA loading its own operand halves with plain TMA
// (described at its definition); gemm_kernel (M ≤ 128) is the single-CTA form
// below.
//
// Design (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: 128-byte-swizzled 128×64 A and 256×64 B tiles
//               into a 4-stage shared-memory ring (mbarrier full/empty pairs);
//   warp 1      MMA issuer: tcgen05.mma cta_group::1 M=128 N=256 K=16 from
//               shared-memory descriptors into one of two TMEM accumulators;
//   warp 2      TMEM allocator (512 columns = two 128×256 fp32 accumulators);
//   warps 4-7   epilogue: tcgen05.ld of the finished accumulator (each warp its
//               32-lane quarter), activation math, outputs staged through a
//               per-warp shared-memory buffer and stored as whole 128-byte
//               lines, so the epilogue of tile t overlaps the MMAs of tile t+1.
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
// Epilogue staging: two 32-row × 128-byte buffers for each of the 4 epilogue
// warps, after the 256-byte barrier block.
constexpr int EPI_STAGE_BYTES = 32 * 128;
constexpr int EPI_WARP_BYTES = 2 * EPI_STAGE_BYTES;
constexpr int EPI_SMEM_BYTES = 4 * EPI_WARP_BYTES;
constexpr size_t SMEM_BYTES = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + 256 + EPI_SMEM_BYTES;

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
  // > 0: a K-major A operand is split along M into chunks of this many rows,
  // chunk j read through maps[seg.map_a + j] (the SP all-gather fused into the
  // loads: every 128-row block lies inside one chunk).
  int32_t a_chunk_rows;
  int32_t a_nchunks;
  int32_t pad1;
  unsigned* status;
  uint64_t timeout_ns;
  EpiParams epi;
};

// Tile t of an mt × nt grid per partial, in groups of GROUP_M rows.
__device__ __forceinline__ void decode_tile_grid(int t, int mt, int nt, int& part, int& mb, int& nb) {
  const int per_part = mt * nt;
  part = t / per_part;
  const int r = t - part * per_part;
  const int span = GROUP_M * nt;
  const int g = r / span;
  const int first_m = g * GROUP_M;
  const int gsz = min(mt - first_m, GROUP_M);
  const int rr = r - g * span;
  mb = first_m + rr % gsz;
  nb = rr / gsz;
}
__device__ __forceinline__ void decode_tile(int t, const Params& p, int& part, int& mb, int& nb) {
  decode_tile_grid(t, p.mt, p.nt, part, mb, nb);
}

// ---------------------------------------------------------------- epilogues
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// Output staging.  After tcgen05.ld a lane holds one row, so storing straight
// from registers makes every warp store touch 32 rows × 16 bytes (32 lines).
// Instead lane r puts its row's 16-byte units u of a 128-byte line segment into
// slot u ^ (r & 7) of row r of a 32 × 128-byte buffer (conflict-free: the 8
// lanes of a quarter-warp hit 8 different slots), and the flush reads it back
// with 8 consecutive lanes on one row, so each warp store writes 4 whole lines.
__device__ __forceinline__ void stage_put(uint32_t buf, int lane, int unit, uint4 v) {
  sts128(buf + static_cast<uint32_t>(lane) * 128u + (static_cast<uint32_t>(unit ^ (lane & 7)) << 4), v);
}
// Writes the staged line segments of rows m0 .. m0 + 31: row m's segment starts
// at byte address line(m); rows at or past M and units at or past `units` are
// skipped.
template <typename LineFn>
__device__ __forceinline__ void stage_flush(uint32_t buf, int lane, int64_t m0, int64_t M, int units, LineFn line) {
  __syncwarp();
  const int u = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    const uint4 v = lds128(buf + static_cast<uint32_t>(r) * 128u + (static_cast<uint32_t>(u ^ (r & 7)) << 4));
    const int64_t m = m0 + r;
    if (m < M && u < units) *reinterpret_cast<uint4*>(line(m) + u * 16) = v;
  }
  __syncwarp();
}
// The read counterpart: loads the 128-byte line segments of rows m0 .. m0 + 31
// (row m's at byte address line(m), 8 lanes per row, rows at or past M and
// units at or past `units` read as zero) into the buffer in the same layout,
// for stage_get to hand each lane its own row's units.
// COHERENT: L2-coherent loads, for data this kernel writes back (main_grad);
// otherwise the read-only path.
template <bool COHERENT = false, typename LineFn>
__device__ __forceinline__ void stage_fill(uint32_t buf, int lane, int64_t m0, int64_t M, int units, LineFn line) {
  const int u = lane & 7;
  uint4 t[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t m = m0 + i * 4 + (lane >> 3);
    if (m < M && u < units) {
      const char* a = line(m) + u * 16;
      t[i] = COHERENT ? __ldcg(reinterpret_cast<const uint4*>(a)) : ldg_nc_v4(a);
    } else {
      t[i] = make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    sts128(buf + static_cast<uint32_t>(r) * 128u + (static_cast<uint32_t>(u ^ (r & 7)) << 4), t[i]);
  }
  __syncwarp();
}
__device__ __forceinline__ uint4 stage_get(uint32_t buf, int lane, int unit) {
  return lds128(buf + static_cast<uint32_t>(lane) * 128u + (static_cast<uint32_t>(unit ^ (lane & 7)) << 4));
}
// 16-byte units of a line segment starting at column n that lie (start) before N
__device__ __forceinline__ int units_before(int64_t N, int64_t n, int cols_per_unit) {
  const int64_t left = N - n;
  if (left <= 0) return 0;
  const int64_t u = (left + cols_per_unit - 1) / cols_per_unit;
  return u >= 8 ? 8 : static_cast<int>(u);
}

// fc2 input gradient epilogue for 8 columns: dU = act'(U) ⊙ dY.  SwiGLU:
// dG = dY·Up·silu'(G) and dUp = dY·silu(G), written to dU's gate and up halves.
// (packed into *gate, and for SwiGLU the up half into *up)
template <int DT>
__device__ __forceinline__ void epi_dact8(const EpiParams& e, const float* dy, uint4 u_raw, uint4 up_raw,
                                          uint4* gate, uint4* upo) {
  float u[8], r[8];
  unpack8<DT>(u_raw, u);
  if (e.act == ACT_SWIGLU) {
    float up[8], r2[8];
    unpack8<DT>(up_raw, up);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float sg = sigmoid_f<false>(u[i]);
      r[i] = dy[i] * up[i] * (sg * (1.0f + u[i] * (1.0f - sg)));
      r2[i] = dy[i] * (u[i] * sg);
    }
    *gate = pack8<DT>(r);
    *upo = pack8<DT>(r2);
    return;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = dy[i] * act_grad<false>(e.act, u[i]);
  *gate = pack8<DT>(r);
}

// L2 prefetch of the saved U row segment a fc2-input-gradient tile will read,
// issued before the epilogue waits for the accumulator.
template <int TN>
__device__ __forceinline__ void epi_prefetch_aux(const Params& p, int64_t m, int nb, int elem_bytes) {
  const EpiParams& e = p.epi;
  if (m >= p.M) return;
  if (e.kind == EPI_ACC_F32) {  // the float32 main_grad rows this tile will update
    const char* row = static_cast<const char*>(e.out) + (m * e.ldo + static_cast<int64_t>(nb) * TN) * 4;
    const int64_t left = (p.N - static_cast<int64_t>(nb) * TN) * 4;
#pragma unroll
    for (int b = 0; b < TN * 4 / 128; ++b)
      if (b * 128 < left) prefetch_l2(row + b * 128);
    return;
  }
  if (e.kind != EPI_DACT) return;
  const char* row = static_cast<const char*>(e.aux) + (m * e.ldaux + static_cast<int64_t>(nb) * TN) * elem_bytes;
  const int64_t left = (p.N - static_cast<int64_t>(nb) * TN) * elem_bytes;
#pragma unroll
  for (int b = 0; b < TN * 2 / 128; ++b) {
    if (b * 128 < left) {
      prefetch_l2(row + b * 128);
      if (e.act == ACT_SWIGLU) prefetch_l2(row + e.swiglu_F * elem_bytes + b * 128);
    }
  }
}

// Drains one 128-row × BN-column accumulator (this warp's 32 lanes = rows)
// from tensor memory and runs the epilogue.  All 32 lanes execute the
// tcgen05.ld instructions; rows past M only skip their stores.  `stage` is this
// warp's pair of staging buffers.
template <int DT, int TN>
__device__ __forceinline__ void epilogue_tile(const Params& p, uint32_t trow, int64_t m, int nb, int part,
                                              uint32_t stage) {
  static_assert(TN % 64 == 0, "16-bit outputs are staged in 64-column line segments");
  const EpiParams& e = p.epi;
  const int lane = static_cast<int>(m & 31);  // rows of a warp start at a multiple of 32
  const int64_t m0 = m - lane;
  const uint32_t buf0 = stage, buf1 = stage + EPI_STAGE_BYTES;
  if (p.swiglu_up_row > 0) {
    // SwiGLU fc1, per 64-column segment of the gate half (two 32-column chunks):
    // the gate and up halves of U go out through the two staging buffers, then
    // Y = silu(gate) · up through the first.
    static_assert(TN % 128 == 0, "SwiGLU tiles hold whole 64-column gate and up segments");
    using T = typename Storage<DT>::T;
    constexpr int64_t ES = static_cast<int64_t>(sizeof(T));
    char* ubase = static_cast<char*>(e.out);
    char* ybase = static_cast<char*>(e.out2);
#pragma unroll 1
    for (int sg = 0; sg < TN / 128; ++sg) {
      const int64_t nl = static_cast<int64_t>(nb) * (TN / 2) + sg * 64;
      const int units = units_before(p.N, nl, 8);
      uint4 yk[8];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float g[32], up[32];
        tmem_ld32(trow + (2 * sg + half) * 32, g);
        tmem_ld32(trow + TN / 2 + (2 * sg + half) * 32, up);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          stage_put(buf0, lane, half * 4 + j, pack8<DT>(g + 8 * j));
          stage_put(buf1, lane, half * 4 + j, pack8<DT>(up + 8 * j));
          float a[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float x = g[8 * j + i];
            a[i] = x * sigmoid_f<false>(x) * up[8 * j + i];
          }
          yk[half * 4 + j] = pack8<DT>(a);
        }
      }
      stage_flush(buf0, lane, m0, p.M, units, [&](int64_t mm) { return ubase + (mm * e.ldo + nl) * ES; });
      stage_flush(buf1, lane, m0, p.M, units,
                  [&](int64_t mm) { return ubase + (mm * e.ldo + e.swiglu_F + nl) * ES; });
#pragma unroll
      for (int j = 0; j < 8; ++j) stage_put(buf0, lane, j, yk[j]);
      stage_flush(buf0, lane, m0, p.M, units, [&](int64_t mm) { return ybase + (mm * e.ldo2 + nl) * ES; });
    }
    return;
  }
  if (e.kind == EPI_DACT) {
    // Per 64-column segment: the saved U (and for SwiGLU the up half) is read as
    // whole lines through the staging buffers, each lane takes its row's units,
    // and the buffers are then reused to stage dU.
    using T = typename Storage<DT>::T;
    const bool swi = e.act == ACT_SWIGLU;
    const int64_t nbase = static_cast<int64_t>(nb) * TN;
    const char* ubase = static_cast<const char*>(e.aux);
    char* obase = static_cast<char*>(e.out);
    constexpr int64_t ES = static_cast<int64_t>(sizeof(T));
#pragma unroll 1
    for (int sg = 0; sg < TN / 64; ++sg) {
      const int64_t nl = nbase + sg * 64;
      const int units = units_before(p.N, nl, 8);
      stage_fill(buf0, lane, m0, p.M, units, [&](int64_t mm) { return ubase + (mm * e.ldaux + nl) * ES; });
      if (swi)
        stage_fill(buf1, lane, m0, p.M, units,
                   [&](int64_t mm) { return ubase + (mm * e.ldaux + e.swiglu_F + nl) * ES; });
      uint4 ug[8], uu[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        ug[j] = stage_get(buf0, lane, j);
        uu[j] = swi ? stage_get(buf1, lane, j) : make_uint4(0, 0, 0, 0);
      }
      __syncwarp();  // every lane has its units before the buffers take dU
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[32];
        tmem_ld32(trow + (2 * sg + half) * 32, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 g, u2;
          epi_dact8<DT>(e, v + 8 * j, ug[half * 4 + j], uu[half * 4 + j], &g, &u2);
          stage_put(buf0, lane, half * 4 + j, g);
          if (swi) stage_put(buf1, lane, half * 4 + j, u2);
        }
      }
      stage_flush(buf0, lane, m0, p.M, units, [&](int64_t mm) { return obase + (mm * e.ldo + nl) * ES; });
      if (swi)
        stage_flush(buf1, lane, m0, p.M, units,
                    [&](int64_t mm) { return obase + (mm * e.ldo + e.swiglu_F + nl) * ES; });
    }
    return;
  }
  if (e.kind == EPI_ACC_F32) {
    // main_grad += C, one 32-column (128-byte) line segment at a time: the
    // segment is read as whole lines with L2-coherent loads (this kernel writes
    // it back), each lane adds its row's accumulator values in place, and the
    // segment is written back as whole lines.
    char* base = static_cast<char*>(e.out);
    const int64_t nbase = static_cast<int64_t>(nb) * TN;
#pragma unroll 1
    for (int c = 0; c < TN / 32; ++c) {
      const int64_t nl = nbase + c * 32;
      const int units = units_before(p.N, nl, 4);
      auto line = [&](int64_t mm) { return base + (mm * e.ldo + nl) * 4; };
      stage_fill<true>(buf0, lane, m0, p.M, units, line);
      float v[32];
      tmem_ld32(trow + c * 32, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint4 o = stage_get(buf0, lane, j);
        o.x = __float_as_uint(__uint_as_float(o.x) + v[4 * j]);
        o.y = __float_as_uint(__uint_as_float(o.y) + v[4 * j + 1]);
        o.z = __float_as_uint(__uint_as_float(o.z) + v[4 * j + 2]);
        o.w = __float_as_uint(__uint_as_float(o.w) + v[4 * j + 3]);
        stage_put(buf0, lane, j, o);
      }
      stage_flush(buf0, lane, m0, p.M, units, line);
    }
    return;
  }
  const int64_t nbase = static_cast<int64_t>(nb) * TN;
  if (e.kind == EPI_F32) {
    // float32 partials: a 32-column chunk is one 128-byte line segment
    char* base = static_cast<char*>(e.out) + static_cast<int64_t>(p.part_base + part) * e.part_stride * 4;
#pragma unroll 1
    for (int c = 0; c < TN / 32; ++c) {
      float v[32];
      tmem_ld32(trow + c * 32, v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        stage_put(buf0, lane, j,
                  make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]),
                             __float_as_uint(v[4 * j + 3])));
      const int64_t nl = nbase + c * 32;
      stage_flush(buf0, lane, m0, p.M, units_before(p.N, nl, 4),
                  [&](int64_t mm) { return base + (mm * e.ldo + nl) * 4; });
    }
    return;
  }
  if (e.kind == EPI_STORE || e.kind == EPI_ACT) {
    using T = typename Storage<DT>::T;
    const bool act = e.kind == EPI_ACT;
#pragma unroll 1
    for (int c = 0; c < TN / 32; ++c) {
      float v[32];
      tmem_ld32(trow + c * 32, v);
      const int half = c & 1;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        stage_put(buf0, lane, half * 4 + j, pack8<DT>(v + 8 * j));
        if (act) {
          float a[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) a[i] = act_fwd<false>(e.act, v[8 * j + i]);
          stage_put(buf1, lane, half * 4 + j, pack8<DT>(a));
        }
      }
      if (half) {
        const int64_t nl = nbase + (c - 1) * 32;
        const int units = units_before(p.N, nl, 8);
        if (e.kind == EPI_STORE && e.scatter) {
          stage_flush(buf0, lane, m0, p.M, units, [&](int64_t mm) {
            const int64_t sh = mm / e.rows_per_shard;
            return static_cast<char*>(e.shard[sh]) + ((mm - sh * e.rows_per_shard) * e.ldo + nl) * static_cast<int64_t>(sizeof(T));
          });
        } else {
          char* base = static_cast<char*>(e.out);
          stage_flush(buf0, lane, m0, p.M, units,
                      [&](int64_t mm) { return base + (mm * e.ldo + nl) * static_cast<int64_t>(sizeof(T)); });
        }
        if (act) {
          char* base2 = static_cast<char*>(e.out2);
          stage_flush(buf1, lane, m0, p.M, units,
                      [&](int64_t mm) { return base2 + (mm * e.ldo2 + nl) * static_cast<int64_t>(sizeof(T)); });
        }
      }
    }
    return;
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
              if (p.a_chunk_rows > 0) {
                // rows past M (last tile) read the last chunk out of range: zero fill
                const int m_off = mb * BM;
                const int j = min(m_off / p.a_chunk_rows, p.a_nchunks - 1);
                tma_load_2d(sa, ma + j, fb, k0, m_off - j * p.a_chunk_rows);
              } else {
                tma_load_2d(sa, ma, fb, k0, mb * BM);
              }
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
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      int part, mb, nb;
      decode_tile(t, p, part, mb, nb);
      const int acc = it & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
      const int64_t m = static_cast<int64_t>(mb) * BM + q * 32 + lane;
      epi_prefetch_aux<BN>(p, m, nb, DT == DT_F32 ? 4 : 2);
      const bool ok = mbar_wait_bounded(tfull0 + 8u * acc, acc_phase, abort_flag, p.status, p.timeout_ns);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      epilogue_tile<DT, BN>(p, trow, m, nb, part,
                            smem_u32(smem + STAGES * STAGE_BYTES + 256) + static_cast<uint32_t>(q * EPI_WARP_BYTES));
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

// ---------------------------------------------------------------- 2-SM kernel
// A CTA pair (cluster of 2) computes one 256×256 tile with tcgen05.mma
// .cta_group::2 (M = 256, N = 256, K = 16), issued by the even CTA.  Each CTA
// loads only its half of A (128 rows) and its half of B (128 rows of the
// 256-wide N tile) — half the L2→SM traffic per FLOP of the 1-SM kernel — into
// a 6-stage ring of 32 KB stages; both CTAs' TMA copies complete on the even
// CTA's "full" barrier, and the MMA commits are multicast to both CTAs' "empty"
// and "accumulator full" barriers.  Each CTA's tensor memory holds its 128 rows
// of both 256-column accumulators; both epilogues release an accumulator by
// arriving on the even CTA's "accumulator empty" barrier.
constexpr int PAIR_STAGES = 6;
constexpr int HALF_M = BM;      // rows of A per CTA
constexpr int PA_BYTES = HALF_M * BK * 2;  // 16 KB
constexpr int PB_BYTES = 128 * BK * 2;     // 16 KB: room for up to 128 B rows per CTA
constexpr int PSTAGE_BYTES = PA_BYTES + PB_BYTES;
constexpr int PAIR_NUM_BARS = 2 * PAIR_STAGES + 5;
constexpr size_t PAIR_SMEM_BYTES = 1024 + static_cast<size_t>(PAIR_STAGES) * PSTAGE_BYTES + 256 + EPI_SMEM_BYTES;

// TN: N extent of the pair's tile; each CTA holds TN/2 rows of B.
// Pair slot q (the q-th cluster of 2) computes the tiles t = q, q + S, q + 2S, …
// (S slots).  Every CTA loads its own 128 A rows and TN/2 B rows: no operand
// is shared between clusters, so every copy stays inside its own pair.
template <int DT, bool A_MN, bool B_MN, int TN>
__global__ void __launch_bounds__(THREADS, 1) gemm_pair_kernel(const __grid_constant__ Params p) {
  constexpr int HALF_N = TN / 2;
  // bytes of one stage (both CTAs): A halves + B halves; an MN-major B half is
  // two 64-column boxes even when TN/2 = 96
  constexpr uint32_t CTA_STAGE_TX = PA_BYTES + (B_MN ? 2 * MN_BOX_BYTES : HALF_N * BK * 2);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + PAIR_STAGES * PA_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PAIR_STAGES * PSTAGE_BYTES);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + PAIR_STAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * PAIR_STAGES);
  const uint32_t tempty0 = smem_u32(bars + 2 * PAIR_STAGES + 2);
  const uint32_t drain_bar = smem_u32(bars + 2 * PAIR_STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + PAIR_NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // within the pair; 0 issues the pair's MMAs
  constexpr uint32_t lead = 0u;              // cluster rank of the pair's even CTA
  const bool leader = rank == 0;
  constexpr uint16_t pair_mask = 0x3u;       // both CTAs of the pair
  auto decode = [&](int t, int& part, int& mb, int& nb) { decode_tile(t, p, part, mb, nb); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < PAIR_STAGES; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);  // the pair's MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8u * a, 1);
      mbar_init(tempty0 + 8u * a, 8);  // 4 epilogue warps in each of the 2 CTAs
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int slot = static_cast<int>(cluster_id_x());
  const int nslots = static_cast<int>(gridDim.x >> 1);
  const int num_tiles = p.mt * p.nt * p.nparts;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      for (int s = p.seg_begin[0]; s < p.seg_begin[p.nparts]; ++s) {
        tma_prefetch_map(&p.maps[p.segs[s].map_a]);
        tma_prefetch_map(&p.maps[p.segs[s].map_b]);
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      bool ok = true;
      for (int t = slot; ok && t < num_tiles; t += nslots) {
        int part, mb, nb;
        decode(t, part, mb, nb);
        const int m_off = mb * (2 * HALF_M) + static_cast<int>(rank) * HALF_M;
        int n_row;  // first B row (K-major) / column (MN-major) this CTA loads
        if (p.swiglu_up_row > 0)
          n_row = (leader ? 0 : p.swiglu_up_row) + nb * HALF_N;  // gate half / up half
        else
          n_row = nb * TN + static_cast<int>(rank) * HALF_N;
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
            const uint32_t fb_local = full0 + 8u * stage;
            const uint32_t fb = mapa_shared(fb_local, lead);  // the pair's even-CTA barrier
            if (leader) mbar_arrive_expect_tx(fb_local, 2 * CTA_STAGE_TX);
            const uint32_t sa = smem_u32(smem_a + stage * PA_BYTES);
            const uint32_t sb = smem_u32(smem_b + stage * PB_BYTES);
            const int k0 = kb * BK;
            if constexpr (!A_MN) {
              if (p.a_chunk_rows > 0) {
                // rows past M (last tile) read the last chunk out of range: zero fill
                const int j = min(m_off / p.a_chunk_rows, p.a_nchunks - 1);
                tma_load_2d_pair(sa, ma + j, fb, k0, m_off - j * p.a_chunk_rows);
              } else
                tma_load_2d_pair(sa, ma, fb, k0, m_off);
            } else {
              tma_load_2d_pair(sa, ma, fb, m_off, k0);
              tma_load_2d_pair(sa + MN_BOX_BYTES, ma, fb, m_off + 64, k0);
            }
            if constexpr (!B_MN) {
              tma_load_2d_pair(sb, mbp, fb, k0, n_row);
            } else {
              tma_load_2d_pair(sb, mbp, fb, n_row, k0);
              tma_load_2d_pair(sb + MN_BOX_BYTES, mbp, fb, n_row + 64, k0);
            }
            issued_mask |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == PAIR_STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // Let copies in flight land before the CTA exits.  The even CTA can watch
        // its full barriers; the odd CTA's copies complete there too, so it waits
        // a fixed time instead.
        if (leader) {
          for (int s = 0; s < PAIR_STAGES; ++s)
            if ((issued_mask >> s) & 1u)
              (void)mbar_wait_bounded(full0 + 8u * s, (issued_phase >> s) & 1u, nullptr, nullptr, p.timeout_ns);
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = make_idesc_f16(DT == DT_BF16, A_MN, B_MN, 2 * HALF_M, TN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = slot; ok && t < num_tiles; t += nslots, ++it) {
        int part, mb, nb;
        decode(t, part, mb, nb);
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
            const uint32_t sa = smem_u32(smem_a + stage * PA_BYTES);
            const uint32_t sb = smem_u32(smem_b + stage * PB_BYTES);
#pragma unroll
            for (int ks = 0; ks < BK / UMMA_K; ++ks) {
              const uint64_t ad = A_MN ? make_sdesc_sw128(sa + ks * 2048u, MN_BOX_BYTES, 1024u)
                                       : make_sdesc_sw128(sa + ks * 32u, 16u, 1024u);
              const uint64_t bd = B_MN ? make_sdesc_sw128(sb + ks * 2048u, MN_BOX_BYTES, 1024u)
                                       : make_sdesc_sw128(sb + ks * 32u, 16u, 1024u);
              tc_mma_f16_pair(d_tmem, ad, bd, idesc, accumulate);
              accumulate = 1u;
            }
            tc_commit_pair_mc(empty0 + 8u * stage, pair_mask);  // frees the stage in both CTAs
            if (++stage == PAIR_STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(tfull0 + 8u * acc, pair_mask);  // both CTAs' accumulator halves ready
      }
      if (!ok) {
        tc_commit_pair_mc(drain_bar, static_cast<uint16_t>(1u << lead));
        (void)mbar_wait_bounded(drain_bar, 0u, nullptr, nullptr, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const uint32_t tempty_leader = mapa_shared(tempty0, lead);
    int it = 0;
    for (int t = slot; t < num_tiles; t += nslots, ++it) {
      int part, mb, nb;
      decode(t, part, mb, nb);
      const int acc = it & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
      const int64_t m = static_cast<int64_t>(mb) * (2 * HALF_M) + static_cast<int64_t>(rank) * HALF_M + q * 32 + lane;
      epi_prefetch_aux<TN>(p, m, nb, DT == DT_F32 ? 4 : 2);
      const bool ok = mbar_wait_bounded(tfull0 + 8u * acc, acc_phase, abort_flag, p.status, p.timeout_ns);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      epilogue_tile<DT, TN>(p, trow, m, nb, part,
                            smem_u32(smem + PAIR_STAGES * PSTAGE_BYTES + 256) + static_cast<uint32_t>(q * EPI_WARP_BYTES));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * acc);
    }
  }

  tc_fence_before();
  cluster_sync_all();  // the pair's MMAs and cross-CTA arrivals are all done
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
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

// mode 0: one CTA per tile; 1: CTA pairs (clusters of 2).
template <int DT, bool A_MN, bool B_MN, int TN>
static int launch_one(const Params& p, int64_t tiles, int mode, cudaStream_t st, const DeviceInfo& dev) {
  static std::mutex mu;
  static uint64_t attr_gen[64][2] = {};  // the device context the attributes were set in
  static int max_clusters[64][2] = {};
  auto* k1 = gemm_kernel<DT, A_MN, B_MN>;
  auto* kp = gemm_pair_kernel<DT, A_MN, B_MN, TN>;
  const unsigned csize = 2u;
  int clusters = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    const int d = (dev.device >= 0 && dev.device < 64) ? dev.device : 0;
    if (attr_gen[d][mode] != dev.generation) {
      const cudaError_t e =
          mode ? cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(PAIR_SMEM_BYTES))
               : cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
      if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
      if (mode) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = csize;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(csize * static_cast<unsigned>(std::max(1, dev.num_sms / static_cast<int>(csize))));
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = PAIR_SMEM_BYTES;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        const cudaError_t e2 = cudaOccupancyMaxActiveClusters(&n, kp, &cfg);
        if (e2 != cudaSuccess || n <= 0)
          return set_error(TPMLP_ERR_CUDA, std::string("cudaOccupancyMaxActiveClusters: ") + cudaGetErrorString(e2));
        max_clusters[d][mode] = n;
      }
      attr_gen[d][mode] = dev.generation;
    }
    clusters = max_clusters[d][mode];
  }
  if (mode == 0) {
    const int grid = static_cast<int>(std::min<int64_t>(tiles, dev.num_sms));
    k1<<<grid, THREADS, SMEM_BYTES, st>>>(p);
  } else {
    // pair slots: at most the resident clusters of 2
    const int slots = static_cast<int>(std::min<int64_t>(tiles, clusters));
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(csize * static_cast<unsigned>(slots));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = PAIR_SMEM_BYTES;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kp, p);
    if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("2-SM GEMM launch: ") + cudaGetErrorString(e));
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(TPMLP_ERR_CUDA, std::string("tensor-core GEMM launch: ") + cudaGetErrorString(e));
  return TPMLP_OK;
}

template <int DT, int TN>
static int dispatch_tn(const Params& p, int64_t tiles, int mode, cudaStream_t st, const DeviceInfo& dev, bool a_mn,
                       bool b_mn) {
  if (!a_mn && !b_mn) return launch_one<DT, false, false, TN>(p, tiles, mode, st, dev);
  if (!a_mn && b_mn) return launch_one<DT, false, true, TN>(p, tiles, mode, st, dev);
  if (a_mn && b_mn) return launch_one<DT, true, true, TN>(p, tiles, mode, st, dev);
  return set_error(TPMLP_ERR_UNSUPPORTED, "MN-major A with K-major B is not instantiated");
}

template <int DT>
static int dispatch(const Params& p, int64_t tiles, int mode, int tn, cudaStream_t st, const DeviceInfo& dev,
                    bool a_mn, bool b_mn) {
  (void)tn;
  return dispatch_tn<DT, BN>(p, tiles, mode, st, dev, a_mn, b_mn);
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
  const bool chunked = g.a_chunk_rows > 0;
  if (chunked && (g.a_mn || g.a_chunk_rows % BM != 0 || g.a_chunks.empty() ||
                  static_cast<int64_t>(g.a_chunks.size()) * g.a_chunk_rows != g.M))
    return set_error(TPMLP_ERR_UNSUPPORTED, "chunked A needs K-major chunks of a multiple of 128 rows covering M");

  // CTA pairs (256-row tiles) whenever there is more than one 128-row block.
  const bool pair = g.M > BM;
  // N tile of the pair kernel.  (A 192-wide variant that trims the last wave of
  // N = h GEMMs measured slower per tile than it saved, so one width is used.)
  const int tn = BN;
  Params p;
  memset(&p, 0, sizeof(p));
  p.M = static_cast<int32_t>(g.M);
  p.N = static_cast<int32_t>(g.N);
  p.mt = static_cast<int32_t>((g.M + (pair ? 2 * BM : BM) - 1) / (pair ? 2 * BM : BM));
  const int tile_n = swiglu ? tn / 2 : tn;
  p.nt = static_cast<int32_t>((g.N + tile_n - 1) / tile_n);
  const int mode = pair ? 1 : 0;
  const uint32_t a_box_rows = static_cast<uint32_t>(BM);  // K-major A: one 128-row box per CTA
  const uint32_t b_box_rows = static_cast<uint32_t>(pair ? tn / 2 : (swiglu ? BN / 2 : BN));
  p.swiglu_up_row = static_cast<int32_t>(g.swiglu_up_row);
  p.a_chunk_rows = chunked ? static_cast<int32_t>(g.a_chunk_rows) : 0;
  p.a_nchunks = chunked ? static_cast<int32_t>(g.a_chunks.size()) : 0;
  p.status = dev->status;
  p.timeout_ns = wait_timeout_ns();
  p.epi = g.epi;

  // Launch batches: consecutive partials whose segments fit the parameter block.
  int seg_i = 0;
  const int nseg = static_cast<int>(g.segs.size());
  int part = 0;
  while (part < g.nparts) {
    int nparts = 0, nsegs = 0, nmaps = 0;
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
      const int chunks = chunked ? static_cast<int>(g.a_chunks.size()) : 1;
      if (nmaps + cnt * (chunks + 1) > MAX_MAPS) {
        if (nparts == 0) return set_error(TPMLP_ERR_UNSUPPORTED, "too many tensor maps in one partial");
        break;
      }
      for (int c = 0; c < cnt; ++c) {
        const GemmSeg& s = g.segs[seg_i + nsegs + c];
        if (s.k <= 0 || s.k >= (1ll << 31)) return set_error(TPMLP_ERR_INVALID_ARG, "bad K segment");
        const int idx = nsegs + c;
        Seg& d = p.segs[idx];
        d.k_len = static_cast<int32_t>(s.k);
        d.map_a = nmaps;
        if (chunked) {
          for (int j = 0; j < chunks; ++j) {
            rc = make_map(&p.maps[nmaps++], g.dtype, g.a_chunks[j], s.k, g.a_chunk_rows, g.lda, BK, a_box_rows);
            if (rc != TPMLP_OK) return rc;
          }
        } else if (!g.a_mn) {
          rc = make_map(&p.maps[nmaps++], g.dtype, s.a, s.k, g.M, g.lda, BK, a_box_rows);
        } else {
          rc = make_map(&p.maps[nmaps++], g.dtype, s.a, g.M, s.k, g.lda, 64, BK);
        }
        if (rc != TPMLP_OK) return rc;
        d.map_b = nmaps;
        if (!g.b_mn)
          rc = make_map(&p.maps[nmaps++], g.dtype, s.b, s.k, g.b_rows, g.ldb, BK, b_box_rows);
        else
          rc = make_map(&p.maps[nmaps++], g.dtype, s.b, g.N, s.k, g.ldb, 64, BK);
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
    double ksum = 0.0;
    for (int c = 0; c < nsegs; ++c) ksum += static_cast<double>(p.segs[c].k_len);
    const double work = 2.0 * static_cast<double>(g.M) * static_cast<double>(swiglu ? 2 * g.N : g.N) * ksum;
    const int ph = prof_begin(PROF_GEMM_TC, st);
    if (g.dtype == DT_BF16)
      rc = dispatch<DT_BF16>(p, tiles, mode, tn, st, *dev, g.a_mn, g.b_mn);
    else
      rc = dispatch<DT_F16>(p, tiles, mode, tn, st, *dev, g.a_mn, g.b_mn);
    prof_end(ph, work, st);
    if (rc != TPMLP_OK) return rc;
    seg_i += nsegs;
  }
  return TPMLP_OK;
}

}  // namespace tpmlp
