// tcgen05 GEMM for the chunk-sliced projections of the attention layer.
//
// The layer's Q, K, V, O matrices and their projections ("the query, key,
// and value matrices in the transformer layer", talk write-up "Untied
// Ulysses Pushes Llama-3-8B Training to 5 Million Tokens", Q&A paragraph)
// are sliced per head-chunk: a chunk only ever materialises its own heads'
// rows of Q/K/V and its own share of the output projection, accumulated
// into a carried partial result (same write-up, paragraph on intermediate
// buffers: "a partial result is stored").
//
// Kernel shape: persistent CTA pairs (clusters of two, one CTA per SM)
// walking 256x256 output tiles.  CTA r of a pair owns the 128 rows of m
// tile 2 mp + r and loads B slot 2 np + r; the even CTA's thread issues
// tcgen05.mma.cta_group::2 (M=256, N=256, K=16), which takes A and B from
// both CTAs' shared memory and leaves each CTA its own 128 rows of D in its
// TMEM.  Per SM that is one 128x256x16 product per 4 KB of A and 4 KB of B
// read from (and written by TMA into) shared memory, against 12 KB for a
// single-CTA 128x256 product: with both operands in shared memory a single
// CTA is bound by shared-memory bandwidth, a pair reaches the tensor rate.
// K goes in blocks of 64 bf16 (one 128-byte swizzle row) through a TMA ring
// that runs across tile boundaries; both CTAs' copies of a stage complete
// directly on the even CTA's barrier (cta_group::2 copies; a software
// forwarding hop from the odd CTA cost ~900 cycles per stage).  D goes into
// one of two 256-column
// TMEM accumulators while the four epilogue warps of each CTA drain the
// other, so a tile's epilogue overlaps the next tile's main loop.
// Operands are K-major (rows of 64 contiguous K) or MN-major (rows of
// contiguous M/N, 64-wide boxes); both use the same swizzled shared layout
// and differ only in the descriptor.
//
// Fixed reduction order: every output element accumulates its K blocks in
// ascending order inside TMEM; a carried fp32 partial (out32 / dx32) is
// loaded into TMEM before the first MMA so that chunked and unchunked runs
// perform the same fp32 additions in the same order.
//
// dWqkv has K = L tokens but only ((U + 2 Hkv_c) / 2) x (D / 256) pair
// tiles (96 for D = 4096, U = 8 query and 2 KV heads: 1.26 waves of 76
// pairs), so it splits K at k_mid into two work units per tile, each reduced
// (red.global.add.f32) into the zeroed output: 192 units fill the pairs 2.5
// times instead of 1.26.  dWo does the same (80 pair tiles at D = 5120,
// U = 8: a second wave of 4 tiles unsplit).  Two addends into a zero give
// the same bits in either order, and k_mid depends only on L, so the result
// stays deterministic and independent of U.
//
// The carried fp32 partials (out32, dx32) move between global memory and the
// epilogue warps through a swizzled shared staging tile per warp: TMEM gives
// each lane one row, and 16-byte accesses to 32 different rows per warp
// instruction left the carry stream latency-bound; through the tile, each
// global access instruction covers four whole 128-byte rows.
#include <atomic>

#include "sm103_ptx.cuh"

namespace upipe {
namespace {

constexpr int kTile = 128 * 64 * 2;  // one 16 KB operand tile (128 x 64 bf16)

// Shared-memory layout per kind.  The weight-gradient and dx GEMMs read the
// layer's dQ/dK/dV as a pair of bf16 tensors (value and rounding residual)
// and accumulate both products, which keeps ~16 significant bits of the
// fp32 gradients through the sum over tokens.
template <int KIND>
struct Layout {
  static constexpr bool kSplit = (KIND == GK_DWQKV || KIND == GK_DX);
  static constexpr bool kCarryKind = (KIND == GK_OPROJ || KIND == GK_DX || KIND == GK_WGRAD);
  static constexpr int kStages = kSplit ? 4 : (kCarryKind ? 5 : 6);
  static constexpr int kA = kSplit ? 2 * kTile : kTile;
  static constexpr int kB = kTile;  // this CTA's 128-column slot of the pair's 256
  static constexpr int kStage = kA + kB;
  // Carry kinds: kXposeChunks 32 x 32 fp32 staging tiles per epilogue warp
  // (4 KB each), through which the carry rows are transposed so that global
  // accesses are whole 128-byte lines.  The O projection (K = U d, short
  // products) stages a whole 128-column slot so that its carry loads are in
  // flight together; dx hides one chunk at a time behind its longer products.
  static constexpr int kXposeChunks = KIND == GK_DX ? 1 : 4;
  static constexpr int OFF_XPOSE = kStages * kStage;
  static constexpr int OFF_BAR = OFF_XPOSE + (kCarryKind ? 4 * kXposeChunks * 4096 : 0);
  static constexpr int B_FULL = 0;                    // even CTA: both CTAs' copies of the stage landed
  static constexpr int B_EMPTY = kStages;             // the pair's products read the stage
  static constexpr int B_ACC_FULL = 2 * kStages;      // per accumulator: products done
  static constexpr int B_ACC_FREE = 2 * kStages + 2;  // even CTA, per accumulator: both CTAs drained it
  static constexpr int B_DRAIN = 2 * kStages + 4;
  static constexpr int B_COUNT = 2 * kStages + 5;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + B_COUNT * 8;
  static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 8;
  static constexpr int kSmemBytes = OFF_ABORT + 8 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "gemm shared memory");
};
constexpr int kThreads = 192;
constexpr int kGroupM = 16;  // m pairs per group of the tile order
constexpr uint32_t kTmemCols = 512;  // two 256-column accumulators

template <int KIND>
struct Traits;
template <> struct Traits<GK_QKV>   { static constexpr int a_mn = 0, b_mn = 0; };
template <> struct Traits<GK_OPROJ> { static constexpr int a_mn = 0, b_mn = 0; };
template <> struct Traits<GK_DO>    { static constexpr int a_mn = 0, b_mn = 1; };
template <> struct Traits<GK_DWO>   { static constexpr int a_mn = 1, b_mn = 1; };
template <> struct Traits<GK_DWQKV> { static constexpr int a_mn = 1, b_mn = 1; };
template <> struct Traits<GK_DX>    { static constexpr int a_mn = 0, b_mn = 1; };
template <> struct Traits<GK_GU>    { static constexpr int a_mn = 0, b_mn = 0; };
template <> struct Traits<GK_GU_BWD> { static constexpr int a_mn = 0, b_mn = 0; };
template <> struct Traits<GK_NN>    { static constexpr int a_mn = 0, b_mn = 1; };
template <> struct Traits<GK_WGRAD> { static constexpr int a_mn = 1, b_mn = 1; };

// `bar` is the shared::cluster address of the even CTA's stage barrier.
template <int KIND>
__device__ __forceinline__ void load_a(const CUtensorMap* m, const GemmParams& p, uint32_t dst, uint32_t bar,
                                       int mt, int kb) {
  if constexpr (KIND == GK_QKV || KIND == GK_DO || KIND == GK_GU || KIND == GK_GU_BWD || KIND == GK_NN) {
    tma_load_2d_pair(dst, m, bar, kb * 64, mt * 128);
  } else if constexpr (KIND == GK_OPROJ) {
    tma_load_2d_pair(dst, m, bar, p.a_col0 + kb * 64, mt * 128);
  } else if constexpr (KIND == GK_DWO || KIND == GK_WGRAD) {
    tma_load_2d_pair(dst, m, bar, mt * 128, kb * 64);
    tma_load_2d_pair(dst + 8192, m, bar, mt * 128 + 64, kb * 64);
  } else if constexpr (KIND == GK_DWQKV) {
    const int z = p.tab0[mt];
    tma_load_3d_pair(dst, m, bar, 0, kb * 64, z);
    tma_load_3d_pair(dst + 8192, m, bar, 64, kb * 64, z);
    tma_load_3d_pair(dst + kTile, m, bar, 0, kb * 64, z + p.lo_z);
    tma_load_3d_pair(dst + kTile + 8192, m, bar, 64, kb * 64, z + p.lo_z);
  } else {  // GK_DX
    const int z = p.tab0[kb >> 1];
    tma_load_3d_pair(dst, m, bar, (kb & 1) * 64, mt * 128, z);
    tma_load_3d_pair(dst + kTile, m, bar, (kb & 1) * 64, mt * 128, z + p.lo_z);
  }
}

template <int KIND>
__device__ __forceinline__ void load_b(const CUtensorMap* m, const GemmParams& p, uint32_t dst, uint32_t bar,
                                       int nt, int kb) {
  if constexpr (KIND == GK_QKV) {
    tma_load_2d_pair(dst, m, bar, kb * 64, p.tab0[nt] * 128);
  } else if constexpr (KIND == GK_OPROJ) {
    tma_load_2d_pair(dst, m, bar, p.b_col0 + kb * 64, nt * 128);
  } else if constexpr (KIND == GK_GU || KIND == GK_GU_BWD) {
    // B slot 2 np holds gate rows np*128.., slot 2 np + 1 the up rows
    // F + np*128..: each CTA of the pair ends with [g | u] of one f range.
    tma_load_2d_pair(dst, m, bar, kb * 64, ((nt & 1) ? p.b_col0 : 0) + (nt >> 1) * 128);
  } else if constexpr (KIND == GK_DO || KIND == GK_DWO || KIND == GK_DWQKV || KIND == GK_NN || KIND == GK_WGRAD) {
    tma_load_2d_pair(dst, m, bar, p.b_col0 + nt * 128, kb * 64);
    tma_load_2d_pair(dst + 8192, m, bar, p.b_col0 + nt * 128 + 64, kb * 64);
  } else {  // GK_DX
    const int row = p.tab1[kb >> 1] * 128 + (kb & 1) * 64;
    tma_load_2d_pair(dst, m, bar, nt * 128, row);
    tma_load_2d_pair(dst + 8192, m, bar, nt * 128 + 64, row);
  }
}

// Four fp32 additions into global memory, performed at L2.
__device__ __forceinline__ void red_add_global_v4(float* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(__uint_as_float(a)),
               "f"(__uint_as_float(b)), "f"(__uint_as_float(c)), "f"(__uint_as_float(d))
               : "memory");
}

template <int MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk) {
  if constexpr (MN) return sdesc_sw128(base + kk * 2048, 8192, 1024);
  else return sdesc_sw128(base + kk * 32, 16, 1024);
}

// Staging-tile address of 16-byte chunk `chunk` of row `row`: rows of 128 B,
// chunks XOR-swizzled by row & 7, so that a warp writing one row per lane and
// a warp reading four rows of eight lanes each both touch every bank once
// per 128 bytes.
__device__ __forceinline__ uint32_t xpose_addr(uint32_t base, int row, int chunk) {
  return base + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// Carry rows m0 .. m0 + 31 (one per lane), columns col .. col + 31, between
// the fp32 carry in global memory and registers, through the warp's staging
// tile `xs`: global accesses go four rows of 128 B per instruction instead of
// 32 rows of 16 B.  All 32 lanes call these together.
__device__ __forceinline__ void carry_store32(const GemmParams& p, uint32_t xs, int m0, int col,
                                              const uint32_t (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 8; ++q) st_shared_v4(xpose_addr(xs, lane, q), v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = 4 * i + (lane >> 3);
    const uint4 y = ld_shared_v4(xpose_addr(xs, row, lane & 7));
    if (m0 + row < p.M)
      st_global_v4(p.carry + static_cast<int64_t>(m0 + row) * p.N + col + (lane & 7) * 4, y.x, y.y, y.z, y.w);
  }
  __syncwarp();
}

// Starts the copy of carry columns col .. col + 31 of rows m0 .. m0 + 31 into
// staging tile `xs` (asynchronous 16-byte copies, four rows of 128 B per
// warp instruction; rows past M or a missing tile are zero-filled).
__device__ __forceinline__ void carry_fetch32(const GemmParams& p, uint32_t xs, int m0, int col, bool tile_ok) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = 4 * i + (lane >> 3);
    const uint32_t dst = xpose_addr(xs, row, lane & 7);
    if (tile_ok && m0 + row < p.M) {
      const float* src = p.carry + static_cast<int64_t>(m0 + row) * p.N + col + (lane & 7) * 4;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
    } else {
      st_shared_v4(dst, 0u, 0u, 0u, 0u);
    }
  }
}

// After the fetches and a cp.async.wait_all + __syncwarp: lane's row of
// staging tile `xs`.
__device__ __forceinline__ void carry_row32(uint32_t xs, uint32_t (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 y = ld_shared_v4(xpose_addr(xs, lane, q));
    v[4 * q] = y.x;
    v[4 * q + 1] = y.y;
    v[4 * q + 2] = y.z;
    v[4 * q + 3] = y.w;
  }
}

// Writes one 128-column slot of a finished accumulator (TMEM row address
// `trow`, one output row per thread) in the kind's output format; `xs` is
// the warp's staging tile (carry kinds).
template <int KIND>
__device__ __forceinline__ void store_slot(const GemmParams& p, uint32_t trow, int m, int r, int mt, int nt,
                                           bool valid, uint32_t xs) {
  constexpr bool kCarry = Layout<KIND>::kCarryKind;
  if constexpr (KIND == GK_QKV) {
    const int slot = nt;
    __nv_bfloat16* orow =
        static_cast<__nv_bfloat16*>(p.out) + (static_cast<int64_t>(slot) * p.L + m) * kHeadDim;
    const bool rot = slot < p.rope_slots;
    const float2* tab = p.rope + static_cast<int64_t>(m) * 64;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t a[32], b[32];
      tmem_ld32(trow + half * 32, a);
      tmem_ld32(trow + 64 + half * 32, b);
      tmem_ld_wait(a);
      tmem_ld_wait(b);
      float lo[32], hi[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float x0 = __uint_as_float(a[i]);
        const float x1 = __uint_as_float(b[i]);
        if (rot && valid) {
          const float2 cs = tab[half * 32 + i];
          lo[i] = x0 * cs.x - x1 * cs.y;
          hi[i] = x0 * cs.y + x1 * cs.x;
        } else {
          lo[i] = x0;
          hi[i] = x1;
        }
      }
      if (valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          st_global_v4(orow + half * 32 + q * 8, pack_bf16x2(lo[8 * q], lo[8 * q + 1]),
                       pack_bf16x2(lo[8 * q + 2], lo[8 * q + 3]), pack_bf16x2(lo[8 * q + 4], lo[8 * q + 5]),
                       pack_bf16x2(lo[8 * q + 6], lo[8 * q + 7]));
          st_global_v4(orow + 64 + half * 32 + q * 8, pack_bf16x2(hi[8 * q], hi[8 * q + 1]),
                       pack_bf16x2(hi[8 * q + 2], hi[8 * q + 3]), pack_bf16x2(hi[8 * q + 4], hi[8 * q + 5]),
                       pack_bf16x2(hi[8 * q + 6], hi[8 * q + 7]));
        }
      }
    }
  } else if constexpr (KIND == GK_DO) {
    const int slot = nt;
    __nv_bfloat16* orow =
        static_cast<__nv_bfloat16*>(p.out) + (static_cast<int64_t>(slot) * p.L + m) * kHeadDim;
    const __nv_bfloat16* obf = p.o_rows + static_cast<int64_t>(m) * p.ld_o + slot * kHeadDim;
    float dsum = 0.f;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      uint32_t v[32];
      tmem_ld32(trow + c4 * 32, v);
      tmem_ld_wait(v);
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
      if (valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          st_global_v4(orow + c4 * 32 + q * 8, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          const uint4 ov = ld_global_nc_v4(obf + c4 * 32 + q * 8);
          const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dsum = fmaf(bf16_lo(pk[4 * q + e]), bf16_lo(ow[e]), dsum);
            dsum = fmaf(bf16_hi(pk[4 * q + e]), bf16_hi(ow[e]), dsum);
          }
        }
      }
    }
    // LSE/Delta record of this row (padding rows past L get -inf / 0).
    const int n_q64 = (p.L + 63) / 64;
    if (m < n_q64 * 64) {
      float* rec = p.ld_rec + (static_cast<int64_t>(slot) * n_q64 + (m >> 6)) * 128;
      rec[m & 63] = valid ? -p.lse_in[static_cast<int64_t>(slot) * p.L + m] * 1.4426950408889634074f : -INFINITY;
      rec[64 + (m & 63)] = valid ? dsum : 0.f;
    }
  } else {
    // fp32 or carried outputs: OPROJ, DX (carry / final bf16), DWO, DWQKV (fp32).
    float* frow = nullptr;
    __nv_bfloat16* brow = nullptr;
    if constexpr (kCarry) {
      if (p.final_out)
        brow = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(m) * p.ld_out + nt * 128;
      else
        frow = p.carry + static_cast<int64_t>(m) * p.N + nt * 128;
    } else if constexpr (KIND == GK_DWO) {
      frow = static_cast<float*>(p.out) + static_cast<int64_t>(m) * p.ld_out + p.out_col0 + nt * 128;
    } else if constexpr (KIND == GK_NN) {
      brow = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(m) * p.ld_out + nt * 128;
    } else {  // GK_DWQKV
      frow = static_cast<float*>(p.out) + static_cast<int64_t>(p.tab1[mt] * 128 + r) * p.ld_out + nt * 128;
    }
    const bool reduce = (KIND == GK_DWQKV || KIND == GK_DWO) && p.k_mid > 0 && p.k_mid < p.k_blocks;
    if constexpr (kCarry) {
      if (!p.final_out) {
        const int m0 = m - (r & 31);
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(trow + c4 * 32, v);
          tmem_ld_wait(v);
          carry_store32(p, xs, m0, nt * 128 + c4 * 32, v);
        }
        return;
      }
    }
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      uint32_t v[32];
      tmem_ld32(trow + c4 * 32, v);
      tmem_ld_wait(v);
      if (valid) {
        if (brow) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_global_v4(brow + c4 * 32 + q * 8,
                         pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                         pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                         pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                         pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
        } else {
          if (reduce) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              red_add_global_v4(frow + c4 * 32 + q * 4, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_global_v4(frow + c4 * 32 + q * 4, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
        }
      }
    }
  }
}

// SwiGLU epilogue of the gate/up GEMM: accumulator columns [0, 128) hold
// g = x Wg^T and [128, 256) u = x Wu^T for features f = 128 np + c of row m.
// Forward: H = silu(g) u.  Backward (dH from in2): H, dG = dH u silu'(g) and
// dU = dH silu(g), with s = sigmoid(g), silu = g s, silu' = s (1 + g (1 - s)).
template <int KIND>
__device__ __forceinline__ void store_gu(const GemmParams& p, uint32_t tacc, int m, int np, bool valid) {
  const int64_t f0 = static_cast<int64_t>(np) * 128;
  __nv_bfloat16* hrow = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(m) * p.ld_out + f0;
#pragma unroll 1
  for (int c4 = 0; c4 < 4; ++c4) {
    uint32_t g[32], u[32];
    tmem_ld32(tacc + c4 * 32, g);
    tmem_ld32(tacc + 128 + c4 * 32, u);
    tmem_ld_wait(g);
    tmem_ld_wait(u);
    if (!valid) continue;
    float dh[32];
    if constexpr (KIND == GK_GU_BWD) {
      const __nv_bfloat16* drow = p.in2 + static_cast<int64_t>(m) * p.ld_in2 + f0 + c4 * 32;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = ld_global_nc_v4(drow + q * 8);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          dh[8 * q + 2 * e] = bf16_lo(w[e]);
          dh[8 * q + 2 * e + 1] = bf16_hi(w[e]);
        }
      }
    }
    uint32_t hp[16], dgp[16], dup[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float hv[2], dg[2], du[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float gv = __uint_as_float(g[2 * i + e]);
        const float uv = __uint_as_float(u[2 * i + e]);
        const float sg = 1.0f / (1.0f + __expf(-gv));
        const float silu = gv * sg;
        hv[e] = silu * uv;
        if constexpr (KIND == GK_GU_BWD) {
          const float d = dh[2 * i + e];
          dg[e] = d * uv * (sg * (1.0f + gv * (1.0f - sg)));
          du[e] = d * silu;
        }
      }
      hp[i] = pack_bf16x2(hv[0], hv[1]);
      if constexpr (KIND == GK_GU_BWD) {
        dgp[i] = pack_bf16x2(dg[0], dg[1]);
        dup[i] = pack_bf16x2(du[0], du[1]);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_global_v4(hrow + c4 * 32 + q * 8, hp[4 * q], hp[4 * q + 1], hp[4 * q + 2], hp[4 * q + 3]);
    if constexpr (KIND == GK_GU_BWD) {
      __nv_bfloat16* grow = p.out2 + static_cast<int64_t>(m) * p.ld_out2 + f0 + c4 * 32;
      __nv_bfloat16* urow = grow + p.b_col0;  // dU block starts at column F
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        st_global_v4(grow + q * 8, dgp[4 * q], dgp[4 * q + 1], dgp[4 * q + 2], dgp[4 * q + 3]);
        st_global_v4(urow + q * 8, dup[4 * q], dup[4 * q + 1], dup[4 * q + 2], dup[4 * q + 3]);
      }
    }
  }
}

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb,
                const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  using Lt = Layout<KIND>;
  constexpr int kStages = Lt::kStages;
  constexpr int OFF_BAR = Lt::OFF_BAR;
  constexpr int B_FULL = Lt::B_FULL, B_EMPTY = Lt::B_EMPTY;
  constexpr int B_ACC_FULL = Lt::B_ACC_FULL, B_ACC_FREE = Lt::B_ACC_FREE, B_DRAIN = Lt::B_DRAIN;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool even = rank == 0;
  // Pair tiles in groups of kGroupM m pairs: within a group the m pair
  // varies fastest, so the ~76 pairs running at once cover at most 16 m
  // pairs by a few n pairs, and both operand slices they read stay in L2
  // (a plain row-major order re-streams all of B once per m pair when B
  // exceeds L2, e.g. the MLP weights or the LM head).
  const int m_pairs = (p.m_tiles + 1) / 2;
  const int n_pairs = (p.n_tiles + 1) / 2;
  const int tiles = m_pairs * n_pairs;
  auto pair_of = [&](int tt, int* mp, int* np) {
    const int span = kGroupM * n_pairs;
    const int first = (tt / span) * kGroupM;
    const int gm = m_pairs - first < kGroupM ? m_pairs - first : kGroupM;
    const int within = tt - (tt / span) * span;
    *mp = first + within % gm;
    *np = within / gm;
  };
  // Work unit t: pair tile t % tiles over K blocks [kb_lo(t), kb_hi(t)).
  const bool ksplit = (KIND == GK_DWQKV || KIND == GK_DWO) && p.k_mid > 0 && p.k_mid < p.k_blocks;
  const int total = ksplit ? 2 * tiles : tiles;
  auto kb_lo = [&](int t) { return ksplit && t >= tiles ? p.k_mid : 0; };
  auto kb_hi = [&](int t) { return ksplit && t < tiles ? p.k_mid : p.k_blocks; };
  const int t0 = blockIdx.x >> 1;
  const int G = gridDim.x >> 1;
  auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lt::OFF_ABORT);
  const WaitCtl w{abort_flag, p.status, p.limit_ns};
  constexpr bool kCarry = Lt::kCarryKind;
  const bool carry_in = kCarry && p.carry_in;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_FULL + s), 2);  // one expect_tx arrival from each CTA's producer
      mbar_init(bar(B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_ACC_FULL + b), 1);
      mbar_init(bar(B_ACC_FREE + b), 8);  // 4 epilogue warps in each CTA
    }
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(sb + Lt::OFF_TMEM_SLOT, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + Lt::OFF_TMEM_SLOT);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&ma);
      tma_prefetch_map(&mb);
      int last[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last[s] = -1;
      int g = 0;  // k blocks issued so far, across tiles
      bool ok = true;
      for (int t = t0; ok && t < total; t += G) {
        int mp, np;
        pair_of(t % tiles, &mp, &np);
        const int mt = 2 * mp + static_cast<int>(rank);
        const int mt_ld = mt < p.m_tiles ? mt : p.m_tiles - 1;  // a missing m tile reloads the last (unused)
        const int ns = 2 * np + static_cast<int>(rank);
        const bool has_b = ns < p.n_tiles;
        for (int kb = kb_lo(t); kb < kb_hi(t); ++kb, ++g) {
          const int s = g % kStages;
          // Polled: the arrival comes from the even CTA's commit, and a
          // suspended try_wait was measured to wake late for it.
          if (!(ok = mbar_spin<true>(bar(B_EMPTY + s), ((g / kStages) & 1) ^ 1, w))) break;
          const uint32_t dst = sb + s * Lt::kStage;
          const uint32_t full = mapa_shared(bar(B_FULL + s), 0);
          mbar_expect_tx_cluster(full, Lt::kA + (has_b ? kTile : 0));
          load_a<KIND>(&ma, p, dst, full, mt_ld, kb);
          if (has_b) load_b<KIND>(&mb, p, dst + Lt::kA, full, ns, kb);
          last[s] = g;
        }
      }
      // Unwinding: every copy of either CTA completes on the even CTA's
      // barriers, so the even CTA waits (bounded) for the stages issued last;
      // the odd CTA stays resident until then (final cluster barrier).  A
      // phase the other CTA never joined does not complete; its 1 s drain
      // limit is far beyond any copy's flight time.
      if (*abort_flag && even) {
        for (int s = 0; s < kStages; ++s)
          if (last[s] >= 0) mbar_wait_drain<true>(bar(B_FULL + s), (last[s] / kStages) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    if (even && lane == 0) {
      // ------------------------------------------- even CTA: pair products
      constexpr uint32_t idesc = idesc_bf16(256, 256, Traits<KIND>::a_mn, Traits<KIND>::b_mn);
      bool ok = true;
      int g = 0;
      int i = 0;
      for (int t = t0; ok && t < total; t += G, ++i) {
        const int b = i & 1;
        const uint32_t acc = tmem + b * 256;
        if (!(ok = mbar_spin<true>(bar(B_ACC_FREE + b), (i >> 1) & 1, w))) break;
        tc_fence_after();
        const int k0 = kb_lo(t);
        for (int kb = k0; kb < kb_hi(t); ++kb, ++g) {
          const int s = g % kStages;
          if (!(ok = mbar_spin<true>(bar(B_FULL + s), (g / kStages) & 1, w))) break;
          tc_fence_after();
          const uint32_t a = sb + s * Lt::kStage;
          const uint32_t bb = a + Lt::kA;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            umma_bf16_pair(acc, operand_desc<Traits<KIND>::a_mn>(a, kk), operand_desc<Traits<KIND>::b_mn>(bb, kk),
                           idesc, (carry_in || kb > k0 || kk > 0) ? 1u : 0u);
          }
          if constexpr (Lt::kSplit) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_pair(acc, operand_desc<Traits<KIND>::a_mn>(a + kTile, kk),
                             operand_desc<Traits<KIND>::b_mn>(bb, kk), idesc, 1u);
          }
          umma_commit_pair(bar(B_EMPTY + s), 0x3);
        }
        if (!ok) break;
        umma_commit_pair(bar(B_ACC_FULL + b), 0x3);
      }
      umma_commit_pair(bar(B_DRAIN), 0x1);
      mbar_wait_drain(bar(B_DRAIN), 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t trow0 = tmem_lane_addr(tmem, quad, 0);
    const uint32_t xs = sb + Lt::OFF_XPOSE + quad * Lt::kXposeChunks * 4096;  // carry kinds only
    const uint32_t acc_free_even = mapa_shared(bar(B_ACC_FREE), 0);
    // Makes accumulator (local tile li) & 1 ready for pair tile t: loads this
    // CTA's rows of the carry when there is one, then tells the even CTA.
    auto prep = [&](int li, int t) {
      if constexpr (kCarry) {
        if (carry_in) {
          int mp, np;
          pair_of(t % tiles, &mp, &np);
          const int mt = 2 * mp + static_cast<int>(rank);
          const int m0 = mt * 128 + quad * 32;  // row of lane 0
          const int nt0 = 2 * np;
          const int nsl = nt0 + 1 < p.n_tiles ? 2 : 1;
          constexpr int kXC = Lt::kXposeChunks;
          for (int j = 0; j < nsl; ++j) {
#pragma unroll 1
            for (int c0 = 0; c0 < 4; c0 += kXC) {
#pragma unroll
              for (int c = 0; c < kXC; ++c)
                carry_fetch32(p, xs + c * 4096, m0, (nt0 + j) * 128 + (c0 + c) * 32, mt < p.m_tiles);
              asm volatile("cp.async.wait_all;" ::: "memory");
              __syncwarp();
#pragma unroll 1
              for (int c = 0; c < kXC; ++c) {
                uint32_t v[32];
                carry_row32(xs + c * 4096, v);
                tmem_st32(trow0 + (li & 1) * 256 + j * 128 + (c0 + c) * 32, v);
              }
              __syncwarp();
            }
          }
          tmem_st_wait();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_free_even + 8 * (li & 1));
    };
    if (t0 < total) prep(0, t0);
    if (t0 + G < total) prep(1, t0 + G);
    bool ok = true;
    int i = 0;
    for (int t = t0; ok && t < total; t += G, ++i) {
      const int b = i & 1;
      int mp, np;
      pair_of(t % tiles, &mp, &np);
      const int mt = 2 * mp + static_cast<int>(rank);
      const int nt0 = 2 * np;
      const int nsl = nt0 + 1 < p.n_tiles ? 2 : 1;
      const int m = mt * 128 + r;
      const bool tile_ok = mt < p.m_tiles;
      const bool valid = tile_ok && m < p.M;
      if (!(ok = warp_wait<true>(bar(B_ACC_FULL + b), (i >> 1) & 1, w))) break;
      tc_fence_after();
      if (tile_ok) {
        if constexpr (KIND == GK_GU || KIND == GK_GU_BWD) {
          store_gu<KIND>(p, trow0 + b * 256, m, np, valid);
        } else {
          for (int j = 0; j < nsl; ++j) {
            const uint32_t trow = trow0 + b * 256 + j * 128;
            store_slot<KIND>(p, trow, m, r, mt, nt0 + j, valid, xs);
          }
        }
      }
      if (t + 2 * G < total) prep(i + 2, t + 2 * G);
    }
    tc_fence_before();
  }

  __syncthreads();
  cluster_sync();  // the even CTA's products are drained; nothing in flight crosses CTAs
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Multiprocessor count of the current device (cached per device; atomic
// entries, so host threads filling the same entry together are well defined).
int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  static std::atomic<int> cached[64];
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int KIND>
cudaError_t launch_kind(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, cudaStream_t s) {
  constexpr int smem = Layout<KIND>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // Persistent: as many pairs as can be resident at once.  A pair must fit
  // inside one GPC, so that is fewer than SMs / 2 when GPCs have odd SM
  // counts; more pairs than that would run as a second wave.
  static std::atomic<int> resident[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (resident[dev].load(std::memory_order_relaxed) <= 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sm_count()), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, gemm_kernel<KIND>, &cfg);
    if (e != cudaSuccess) return e;
    resident[dev].store(n > 0 ? n : 1, std::memory_order_relaxed);
  }
  const int res = resident[dev].load(std::memory_order_relaxed);
  const int tiles = ((p.m_tiles + 1) / 2) * ((p.n_tiles + 1) / 2);
  const int total = ((KIND == GK_DWQKV || KIND == GK_DWO) && p.k_mid > 0 && p.k_mid < p.k_blocks) ? 2 * tiles : tiles;
  const int pairs = total < res ? total : res;
  if (pairs <= 0) return cudaSuccess;
  gemm_kernel<KIND><<<2 * pairs, kThreads, smem, s>>>(a, b, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                        cudaStream_t s) {
  switch (kind) {
    case GK_QKV: return launch_kind<GK_QKV>(a, b, p, s);
    case GK_OPROJ: return launch_kind<GK_OPROJ>(a, b, p, s);
    case GK_DO: return launch_kind<GK_DO>(a, b, p, s);
    case GK_DWO: return launch_kind<GK_DWO>(a, b, p, s);
    case GK_DWQKV: return launch_kind<GK_DWQKV>(a, b, p, s);
    case GK_DX: return launch_kind<GK_DX>(a, b, p, s);
    case GK_GU: return launch_kind<GK_GU>(a, b, p, s);
    case GK_GU_BWD: return launch_kind<GK_GU_BWD>(a, b, p, s);
    case GK_NN: return launch_kind<GK_NN>(a, b, p, s);
    case GK_WGRAD: return launch_kind<GK_WGRAD>(a, b, p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace upipe
