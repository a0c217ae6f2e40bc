// Exact causal attention backward for one head-chunk, tcgen05 + TMEM.
//
// The gradient of softmax attention in closed form: with P = exp(S - LSE),
// dP = dO V^T, Delta_i = sum_k dO_ik O_ik and dS = P * (dP - Delta):
//   dV = P^T dO,  dK = dS^T Q / sqrt(d),  dQ = dS K / sqrt(d).
// The pages fix the formula ("not a new attention formula, but a different
// memory schedule", talk write-up "Untied Ulysses Pushes Llama-3-8B Training
// to 5 Million Tokens", paragraph on intermediate buffers) and the use of
// recomputation in the backward pass (same write-up, paragraph on activation
// checkpointing); the backward schedule below is this library's own.
//
// Two kernels, neither using atomics, so every result has one fixed fp32
// summation order that does not depend on the chunk size U:
//  * dq kernel: one CTA per (query head, 128-query tile) walks its 128-key
//    blocks in ascending order and accumulates dQ in TMEM;
//  * dkdv kernel: one CTA per (KV head, 128-key tile) walks the query heads
//    that read this KV head (ascending) and, for each, the 128-query tiles
//    at or after the key tile (ascending), accumulating dK and dV in TMEM.  When
//    a chunk holds fewer query heads than a KV group (U < g) the partial sums
//    are carried in fp32 between chunks and reloaded into TMEM, which keeps
//    the same order as a single pass over the whole group.
//
// Both kernels have one producer warp loading tiles with TMA, one issuing
// warp per product kind (a single thread issues a tcgen05.mma only about
// every 100 cycles), and compute warps that turn scores into P / dS.  Warp w
// of the compute warps reads TMEM lane quadrant w % 4, so the warps sharing a
// quadrant split its columns.  Shared-memory operand reads run at roughly
// 80-100 B/clk per SM, so the softmax tiles (P^T, dS^T, dS) stay in TMEM and
// feed the products that consume them as TMEM A operands.
#include "sm103_ptx.cuh"

namespace upipe {
namespace {

// Warp roles of the dq kernel (the dkdv kernel has its own, below).  One
// thread issues a tcgen05.mma about every 100 cycles at best, so each product
// kind has its own issuing warp, owning its own accumulators.
constexpr int kComputeWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;    // issues S; allocates TMEM
constexpr int kGradWarp = 10;  // issues dQ, which consumes dS from TMEM
constexpr uint32_t kTmemCols = 512;

// dS row slice of the dq kernel: 32 keys of one query row, paired fp32
// math.  kMask applies the causal mask (only the diagonal tile needs it).
template <bool kMask>
__device__ __forceinline__ void ds_slice(const uint32_t (&sv)[32], const uint32_t (&dv)[32], float sl2, float nlse2,
                                         float dlt, int k0, int qpos, uint32_t (&pk)[16]) {
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  const uint64_t nlx2 = f2_pack(nlse2, nlse2);
  const uint64_t dlx2 = f2_pack(dlt, dlt);
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    float t0, t1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, nlx2), t0, t1);
    float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
    if (kMask) {
      if (k0 + c > qpos) p0 = 0.f;
      if (k0 + c + 1 > qpos) p1 = 0.f;
    }
    const uint64_t d = f2_sub(f2_pack(__uint_as_float(dv[c]), __uint_as_float(dv[c + 1])), dlx2);
    float d0, d1;
    f2_unpack(f2_mul(f2_pack(p0, p1), d), d0, d1);
    pk[c >> 1] = pack_bf16x2(d0, d1);
  }
}

// P^T row slice of the dkdv kernel: 16 queries (columns c0 .. c0 + 15 of
// this warp's 32) of one key row, kept in fp32 for the dS^T phase.  Lane c of
// the warp holds -LSE * log2(e) of the warp's query c in `nl`; kMask zeroes
// queries before the key (the diagonal tile only).
template <bool kMask>
__device__ __forceinline__ void p_slice(const uint32_t (&sv)[16], float nl, int c0, float sl2, int q0, int kpos,
                                        float* pf) {
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    const float l0 = __shfl_sync(0xffffffffu, nl, c0 + c);
    const float l1 = __shfl_sync(0xffffffffu, nl, c0 + c + 1);
    float t0, t1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, f2_pack(l0, l1)), t0, t1);
    float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
    if (kMask) {
      if (q0 + c0 + c < kpos) p0 = 0.f;
      if (q0 + c0 + c + 1 < kpos) p1 = 0.f;
    }
    pf[c] = p0;
    pf[c + 1] = p1;
  }
}

// dS^T row slice of the dkdv kernel: dS = P * (dP - Delta) for 16 queries
// (columns c0 .. c0 + 15), packed bf16.  Lane c holds Delta of query c in `dl`.
__device__ __forceinline__ void dst_slice(const uint32_t (&dv)[16], const float* pf, float dl, int c0,
                                          uint32_t (&dd)[8]) {
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    const float d0 = __shfl_sync(0xffffffffu, dl, c0 + c);
    const float d1 = __shfl_sync(0xffffffffu, dl, c0 + c + 1);
    float s0, s1;
    f2_unpack(f2_mul(f2_pack(pf[c], pf[c + 1]),
                     f2_sub(f2_pack(__uint_as_float(dv[c]), __uint_as_float(dv[c + 1])), f2_pack(d0, d1))),
              s0, s1);
    dd[c >> 1] = pack_bf16x2(s0, s1);
  }
}

// ============================================================== dQ kernel
//
// KV blocks of 128 keys, so every product is an M=128, N=128 tcgen05.mma.
// S = Q K^T goes into one of two TMEM buffers; dP = dO V^T into one buffer
// that the compute warps release as soon as they have read it; the compute
// warps write dS (packed bf16) over the S columns they have read, and
// dQ += dS K takes dS straight from TMEM.  K and V stream through separate
// TMA rings: V is released after dP (two stages suffice), K only after dQ,
// about a block later, so its ring has three.  S, dP and dQ each have their
// own issuing warp.

namespace dq {
constexpr int kTile = 128 * 128 * 2;   // [128][128] bf16 as two 64-column halves
constexpr int kHalf = kTile / 2;
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int OFF_Q = 0;
constexpr int OFF_DO = OFF_Q + kTile;
constexpr int OFF_K = OFF_DO + kTile;              // kKStages
constexpr int OFF_V = OFF_K + kKStages * kTile;    // kVStages
constexpr int OFF_BAR = OFF_V + kVStages * kTile;
enum {
  B_QDO_FULL,
  B_K_FULL,
  B_K_EMPTY = B_K_FULL + kKStages,
  B_V_FULL = B_K_EMPTY + kKStages,
  B_V_EMPTY = B_V_FULL + kVStages,
  B_S_FULL = B_V_EMPTY + kVStages,
  B_S_FREE = B_S_FULL + 2,   // dQ of that buffer done: its S/dS columns free
  B_DS_FULL = B_S_FREE + 2,
  B_DP_FULL = B_DS_FULL + 2,
  B_DP_EMPTY,                // the compute warps have read dP
  B_DQ_DONE,
  B_DRAIN,
  B_DRAIN_G,
  B_DRAIN_P,
  B_COUNT
};
constexpr int OFF_TMEM_SLOT = OFF_BAR + B_COUNT * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 8;
constexpr int kSmemBytes = OFF_ABORT + 8 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "dq kernel shared memory");
constexpr int TM_S = 0, TM_DP = 256, TM_DQ = 384;  // S: two 128-column buffers
// Warps 0-7 compute, 8 producer, 9 issues S, 10 issues dQ, 11 issues dP.
constexpr int kDpWarp = 11;
constexpr int kThreadsDq = 384;
}  // namespace dq

__global__ void __launch_bounds__(dq::kThreadsDq, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                       const __grid_constant__ AttnBwdParams p) {
  using namespace dq;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Heads vary fastest (GQA siblings share K/V blocks in L2); the query
  // blocks with the most KV blocks launch first.
  const int h = static_cast<int>(blockIdx.x) % p.nheads;
  const int qb = static_cast<int>(gridDim.x) / p.nheads - 1 - static_cast<int>(blockIdx.x) / p.nheads;
  const int kz = p.k_z0 + h / p.g_loc;
  const int vz = p.v_z0 + h / p.g_loc;
  const int n_kv = qb + 1;  // causal: 128-key blocks 0 .. qb
  auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  const WaitCtl w{abort_flag, p.status, p.limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QDO_FULL), 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(B_K_FULL + s), 1);
      mbar_init(bar(B_K_EMPTY + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(B_V_FULL + s), 1);
      mbar_init(bar(B_V_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_S_FULL + b), 1);
      mbar_init(bar(B_S_FREE + b), 1);
      mbar_init(bar(B_DS_FULL + b), kComputeWarps);
    }
    mbar_init(bar(B_DP_FULL), 1);
    mbar_init(bar(B_DP_EMPTY), kComputeWarps);
    mbar_init(bar(B_DQ_DONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN_G), 1);
    mbar_init(bar(B_DRAIN_P), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sb + OFF_TMEM_SLOT, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);

  if (warp == kProducerWarp) {
    if (lane == 0) {
      tma_prefetch_map(&mq);
      tma_prefetch_map(&mk);
      tma_prefetch_map(&mv);
      tma_prefetch_map(&mdo);
      mbar_expect_tx(bar(B_QDO_FULL), 2 * kTile);
      tma_load_3d(sb + OFF_Q, &mq, bar(B_QDO_FULL), 0, qb * 128, p.q_z0 + h);
      tma_load_3d(sb + OFF_Q + kHalf, &mq, bar(B_QDO_FULL), 64, qb * 128, p.q_z0 + h);
      tma_load_3d(sb + OFF_DO, &mdo, bar(B_QDO_FULL), 0, qb * 128, p.do_z0 + h);
      tma_load_3d(sb + OFF_DO + kHalf, &mdo, bar(B_QDO_FULL), 64, qb * 128, p.do_z0 + h);
      int last_k[kKStages], last_v[kVStages];
#pragma unroll
      for (int s = 0; s < kKStages; ++s) last_k[s] = -1;
#pragma unroll
      for (int s = 0; s < kVStages; ++s) last_v[s] = -1;
      // Whichever ring has a free stage gets its next block, K first (S(j)
      // needs K(j) before dP(j) needs V(j)).
      int nk = 0, nv = 0;
      Watchdog wd;
      wd.reset();
      bool ok = true;
      while (ok && (nk < n_kv || nv < n_kv)) {
        bool did = false;
        if (nk < n_kv && mbar_test(bar(B_K_EMPTY + nk % kKStages), ((nk / kKStages) & 1) ^ 1)) {
          const int s = nk % kKStages;
          mbar_expect_tx(bar(B_K_FULL + s), kTile);
          tma_load_3d(sb + OFF_K + s * kTile, &mk, bar(B_K_FULL + s), 0, nk * 128, kz);
          tma_load_3d(sb + OFF_K + s * kTile + kHalf, &mk, bar(B_K_FULL + s), 64, nk * 128, kz);
          last_k[s] = nk++;
          did = true;
        }
        if (nv < n_kv && mbar_test(bar(B_V_EMPTY + nv % kVStages), ((nv / kVStages) & 1) ^ 1)) {
          const int s = nv % kVStages;
          mbar_expect_tx(bar(B_V_FULL + s), kTile);
          tma_load_3d(sb + OFF_V + s * kTile, &mv, bar(B_V_FULL + s), 0, nv * 128, vz);
          tma_load_3d(sb + OFF_V + s * kTile + kHalf, &mv, bar(B_V_FULL + s), 64, nv * 128, vz);
          last_v[s] = nv++;
          did = true;
        }
        if (did) wd.reset();
        else ok = wd.alive(w);
      }
      if (*abort_flag) {
        mbar_wait_drain(bar(B_QDO_FULL), 0, p.status);
        for (int s = 0; s < kKStages; ++s)
          if (last_k[s] >= 0) mbar_wait_drain(bar(B_K_FULL + s), (last_k[s] / kKStages) & 1, p.status);
        for (int s = 0; s < kVStages; ++s)
          if (last_v[s] >= 0) mbar_wait_drain(bar(B_V_FULL + s), (last_v[s] / kVStages) & 1, p.status);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // S(j) = Q K(j)^T into buffer j & 1 once K(j) has landed and dQ(j - 2)
      // has released the buffer.
      constexpr uint32_t id_kk = idesc_bf16(128, 128, 0, 0);
      bool ok = mbar_spin(bar(B_QDO_FULL), 0, w);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % kKStages;
        if (!(ok = mbar_spin(bar(B_K_FULL + s), (j / kKStages) & 1, w))) break;
        if (!(ok = mbar_spin(bar(B_S_FREE + (j & 1)), ((j >> 1) & 1) ^ 1, w))) break;
        tc_fence_after();
        const uint32_t ka = sb + OFF_K + s * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_bf16(tmem + TM_S + (j & 1) * 128, sdesc_sw128(sb + OFF_Q + off, 16, 1024),
                    sdesc_sw128(ka + off, 16, 1024), id_kk, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_S_FULL + (j & 1)));
      }
      umma_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0, p.status);
    }
  } else if (warp == kDpWarp) {
    if (lane == 0) {
      // dP(j) = dO V(j)^T once V(j) has landed and dP(j - 1) has been read.
      constexpr uint32_t id_kk = idesc_bf16(128, 128, 0, 0);
      bool ok = mbar_spin(bar(B_QDO_FULL), 0, w);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % kVStages;
        if (!(ok = mbar_spin(bar(B_V_FULL + s), (j / kVStages) & 1, w))) break;
        if (!(ok = mbar_spin(bar(B_DP_EMPTY), (j & 1) ^ 1, w))) break;
        tc_fence_after();
        const uint32_t va = sb + OFF_V + s * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_bf16(tmem + TM_DP, sdesc_sw128(sb + OFF_DO + off, 16, 1024), sdesc_sw128(va + off, 16, 1024), id_kk,
                    kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_DP_FULL));
        umma_commit(bar(B_V_EMPTY + s));
      }
      umma_commit(bar(B_DRAIN_P));
      mbar_wait_drain(bar(B_DRAIN_P), 0, p.status);
    }
  } else if (warp == kGradWarp) {
    if (lane == 0) {
      // dQ(j) += dS(j) K(j) once dS(j) is written; then S buffer j & 1 and
      // K stage j % kKStages are free (S(j) had completed before dS(j) existed).
      constexpr uint32_t id_q = idesc_bf16(128, 128, 0, 1);  // dS from TMEM, K MN-major
      bool ok = true;
      for (int j = 0; ok && j < n_kv; ++j) {
        const int b = j & 1;
        const int s = j % kKStages;
        if (!(ok = mbar_spin(bar(B_DS_FULL + b), (j >> 1) & 1, w))) break;
        tc_fence_after();
        const uint32_t ka = sb + OFF_K + s * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // keys 16 kk .. 16 kk + 15: compute half kk / 4 wrote them at its own
          // 64-column slice of the S buffer
          const uint32_t a = tmem + TM_S + b * 128 + (kk >> 2) * 64 + (kk & 3) * 8;
          umma_bf16_ts(tmem + TM_DQ, a, sdesc_sw128(ka + kk * 2048, kHalf, 1024), id_q, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_S_FREE + b));
        umma_commit(bar(B_K_EMPTY + s));
      }
      if (ok) umma_commit(bar(B_DQ_DONE));
      umma_commit(bar(B_DRAIN_G));
      mbar_wait_drain(bar(B_DRAIN_G), 0, p.status);
    }
  } else {
    // Compute warps: quadrant (warp & 3) of the TMEM lanes = query rows,
    // half (warp >> 2) of the 128 key columns of each block.
    const int quad = warp & 3;
    const int half = warp >> 2;
    const int r = quad * 32 + lane;
    const int qpos = qb * 128 + r;
    const bool valid = qpos < p.L;
    const uint32_t trow = tmem_lane_addr(tmem, quad, 0);
    const float sl2 = p.scale_log2;
    const int n_q64 = (p.L + 63) / 64;
    const float* rec = p.ld + (static_cast<int64_t>(h) * n_q64 + (qpos >> 6)) * 128;
    const float nlse2 = valid ? rec[qpos & 63] : 0.f;  // -LSE * log2(e)
    const float dlt = valid ? rec[64 + (qpos & 63)] : 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      if (!(ok = warp_wait<false, true>(bar(B_S_FULL + b), (j >> 1) & 1, w))) break;
      if (!(ok = warp_wait<false, true>(bar(B_DP_FULL), j & 1, w))) break;
      tc_fence_after();
      const uint32_t ts = trow + TM_S + b * 128 + half * 64;
      uint32_t s0[32], s1[32], d0[32], d1[32];
      tmem_ld32(ts, s0);
      tmem_ld32(ts + 32, s1);
      tmem_ld32(trow + TM_DP + half * 64, d0);
      tmem_ld32(trow + TM_DP + half * 64 + 32, d1);
      tmem_ld_wait(s0);
      tmem_ld_wait(s1);
      tmem_ld_wait(d0);
      tmem_ld_wait(d1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DP_EMPTY));
      const int k0 = j * 128 + half * 64;  // key of this warp's first column
      uint32_t pk0[16], pk1[16];
      if (j == qb) {  // the diagonal block (warp-uniform)
        ds_slice<true>(s0, d0, sl2, nlse2, dlt, k0, qpos, pk0);
        ds_slice<true>(s1, d1, sl2, nlse2, dlt, k0 + 32, qpos, pk1);
      } else {
        ds_slice<false>(s0, d0, sl2, nlse2, dlt, k0, qpos, pk0);
        ds_slice<false>(s1, d1, sl2, nlse2, dlt, k0 + 32, qpos, pk1);
      }
      // dS over the first 32 of the 64 S columns this warp just read.
      tmem_st16(ts, pk0);
      tmem_st16(ts + 16, pk1);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DS_FULL + b));
    }
    if (ok) ok = warp_wait<false, true>(bar(B_DQ_DONE), 0, w);
    if (ok) {
      // Epilogue: this warp writes RoPE pairs (i, i + 64), i in [32 half, 32 half + 32).
      tc_fence_after();
      __nv_bfloat16* out = p.dq + static_cast<int64_t>(qpos) * p.dq_row + static_cast<int64_t>(h) * p.dq_head;
      const float2* tab = p.rope ? p.rope + static_cast<int64_t>(qpos) * 64 : nullptr;
      uint32_t a[32], b[32];
      tmem_ld32(trow + TM_DQ + half * 32, a);
      tmem_ld32(trow + TM_DQ + 64 + half * 32, b);
      tmem_ld_wait(a);
      tmem_ld_wait(b);
      float lo[32], hi[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float x0 = __uint_as_float(a[i]) * p.scale;
        const float x1 = __uint_as_float(b[i]) * p.scale;
        if (tab && valid) {
          const float2 cs = tab[half * 32 + i];
          lo[i] = x0 * cs.x + x1 * cs.y;
          hi[i] = x1 * cs.x - x0 * cs.y;
        } else {
          lo[i] = x0;
          hi[i] = x1;
        }
      }
      if (valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          store8_bf16_split(out + half * 32 + q * 8, lo + 8 * q, p.lo_off);
          store8_bf16_split(out + 64 + half * 32 + q * 8, hi + 8 * q, p.lo_off);
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ============================================================ dK/dV kernel
//
// 128-query tiles, so every product is an M=128, N=128 tcgen05.mma.  TMEM
// holds S^T (128 columns), dP^T (128), dV and dK; with no room for a second
// S^T/dP^T buffer the compute warps work in two phases per tile: P^T as soon
// as S^T has landed (written packed over the S^T columns they read, feeding
// dV while dP^T is still being formed), then dS^T = P^T * (dP^T - Delta)
// over the dP^T columns (feeding dK).  S^T of the next tile is issued as soon
// as dV has consumed P^T, ahead of dK when dS^T is not yet written, so the
// tensor pipe works on it while the compute warps finish dS^T.
// Q/dO tiles stream through a 2-stage TMA ring.  The compute warps read the
// queries' LSE/Delta records straight from global memory (L1-cached, one
// broadcast line per warp): kept out of shared memory, their loads and the
// warps' barrier polls do not queue behind the ring's 64 KB TMA bursts.

namespace dkv {
constexpr int kTile = 128 * 128 * 2;  // K, V, Q or dO tile: [128 rows][128 d]
constexpr int kHalf = kTile / 2;
constexpr int kStages = 2;            // Q/dO ring depth
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + kTile;
constexpr int OFF_Q = OFF_V + kTile;             // kStages stages
constexpr int OFF_DO = OFF_Q + kStages * kTile;
constexpr int OFF_BAR = OFF_DO + kStages * kTile;
enum {
  B_KV_FULL,
  B_QDO_FULL,
  B_QDO_EMPTY = B_QDO_FULL + kStages,
  B_S_FULL = B_QDO_EMPTY + kStages,  // per 64-query half of S^T
  B_P_FULL = B_S_FULL + 2,           // P^T of that half written (its 8 compute warps)
  B_S_FREE = B_P_FULL + 2,           // dV of that half done: its S^T / P^T columns free
  B_DP_FULL = B_S_FREE + 2,
  B_DS_FULL,   // dS^T written (compute warps)
  B_DP_FREE,   // dK done: dP^T / dS^T columns free
  B_CARRY_READY,
  B_DKV_DONE,
  B_DRAIN,
  B_DRAIN_G,
  B_DRAIN_P,
  B_COUNT
};
constexpr int OFF_TMEM_SLOT = OFF_BAR + B_COUNT * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 8;
constexpr int kSmemBytes = OFF_ABORT + 8 + 1024;
constexpr int TM_ST = 0, TM_DPT = 128, TM_DV = 256, TM_DK = 384;
// 16 compute warps: four per TMEM lane quadrant, each owning 32 of the 128
// query columns, so each SM sub-partition has four to hide TMEM and exp2
// latency; then the producer and three MMA-issuing warps (S^T; dV and dK;
// dP^T).
constexpr int kCompute = 16;
constexpr int kProducer = 16;
constexpr int kMma = 17;
constexpr int kGrad = 18;
constexpr int kDpMma = 19;
constexpr int kThreadsKv = 640;
}  // namespace dkv

__global__ void __launch_bounds__(dkv::kThreadsKv, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                         const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                         const __grid_constant__ AttnBwdParams p) {
  using namespace dkv;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Key tile 0 sees every query: the heaviest tiles launch first, KV heads
  // varying fastest.
  const int kb = static_cast<int>(blockIdx.x) / p.nkv;
  const int kv = static_cast<int>(blockIdx.x) % p.nkv;
  const int n_q64 = (p.L + 63) / 64;
  const int n_q128 = (p.L + 127) / 128;
  const int nqt = n_q128 - kb;  // query tiles at or after this key tile
  const int n_it = p.g_loc * nqt;
  auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  const WaitCtl w{abort_flag, p.status, p.limit_ns};
  const bool carry_in = p.carry_in != 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_KV_FULL), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_QDO_FULL + s), 1);
      mbar_init(bar(B_QDO_EMPTY + s), 1);
    }
    for (int hf = 0; hf < 2; ++hf) {
      mbar_init(bar(B_S_FULL + hf), 1);
      mbar_init(bar(B_P_FULL + hf), kCompute / 2);
      mbar_init(bar(B_S_FREE + hf), 1);
    }
    mbar_init(bar(B_DP_FULL), 1);
    mbar_init(bar(B_DS_FULL), kCompute);
    mbar_init(bar(B_DP_FREE), 1);
    mbar_init(bar(B_CARRY_READY), kCompute);
    mbar_init(bar(B_DKV_DONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN_G), 1);
    mbar_init(bar(B_DRAIN_P), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMma) {
    tmem_alloc(sb + OFF_TMEM_SLOT, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);

  if (warp == kProducer) {
    // Q and dO tiles (TMA), both on one barrier per stage.
    if (lane == 0) {
      int last[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last[s] = -1;
      tma_prefetch_map(&mq);
      tma_prefetch_map(&mk);
      tma_prefetch_map(&mv);
      tma_prefetch_map(&mdo);
      mbar_expect_tx(bar(B_KV_FULL), 2 * kTile);
      tma_load_3d(sb + OFF_K, &mk, bar(B_KV_FULL), 0, kb * 128, p.k_z0 + kv);
      tma_load_3d(sb + OFF_K + kHalf, &mk, bar(B_KV_FULL), 64, kb * 128, p.k_z0 + kv);
      tma_load_3d(sb + OFF_V, &mv, bar(B_KV_FULL), 0, kb * 128, p.v_z0 + kv);
      tma_load_3d(sb + OFF_V + kHalf, &mv, bar(B_KV_FULL), 64, kb * 128, p.v_z0 + kv);
      for (int it = 0; it < n_it; ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        const int hl = kv * p.g_loc + it / nqt;
        const int qt = kb + it % nqt;
        if (!mbar_wait(bar(B_QDO_EMPTY + s), ph ^ 1, w)) break;
        mbar_expect_tx(bar(B_QDO_FULL + s), 2 * kTile);
        tma_load_3d(sb + OFF_Q + s * kTile, &mq, bar(B_QDO_FULL + s), 0, qt * 128, p.q_z0 + hl);
        tma_load_3d(sb + OFF_Q + s * kTile + kHalf, &mq, bar(B_QDO_FULL + s), 64, qt * 128, p.q_z0 + hl);
        tma_load_3d(sb + OFF_DO + s * kTile, &mdo, bar(B_QDO_FULL + s), 0, qt * 128, p.do_z0 + hl);
        tma_load_3d(sb + OFF_DO + s * kTile + kHalf, &mdo, bar(B_QDO_FULL + s), 64, qt * 128, p.do_z0 + hl);
        last[s] = it;
      }
      if (*abort_flag) {
        mbar_wait_drain(bar(B_KV_FULL), 0, p.status);
        for (int s = 0; s < kStages; ++s)
          if (last[s] >= 0) mbar_wait_drain(bar(B_QDO_FULL + s), (last[s] / kStages) & 1, p.status);
      }
    }
  } else if (warp == kMma) {
    if (lane == 0) {
      // S^T(i) in two 64-query halves (N=64): half h once the Q/dO stage has
      // landed and dV of half h of tile i - 1 has consumed the P^T there.
      // The halves pipeline independently, which shortens the chain
      // S^T -> P^T -> dV -> next S^T that a single buffer imposes.
      constexpr uint32_t id_s = idesc_bf16(128, 64, 0, 0);
      bool ok = mbar_spin(bar(B_KV_FULL), 0, w);
      for (int it = 0; ok && it < n_it; ++it) {
        const int qs = it % kStages;
        if (!(ok = mbar_spin(bar(B_QDO_FULL + qs), (it / kStages) & 1, w))) break;
        for (int hf = 0; hf < 2; ++hf) {
          if (!(ok = mbar_spin(bar(B_S_FREE + hf), (it & 1) ^ 1, w))) break;
          tc_fence_after();
          const uint32_t bq = sb + OFF_Q + qs * kTile + hf * 64 * 128;  // query rows 64 hf ..
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            umma_bf16(tmem + TM_ST + hf * 64, sdesc_sw128(sb + OFF_K + off, 16, 1024), sdesc_sw128(bq + off, 16, 1024),
                      id_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(bar(B_S_FULL + hf));
        }
      }
      umma_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0, p.status);
    }
  } else if (warp == kDpMma) {
    if (lane == 0) {
      // dP^T(i) = V dO(i)^T once the stage has landed and dK(i - 1) is done.
      constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);
      bool ok = mbar_spin(bar(B_KV_FULL), 0, w);
      for (int it = 0; ok && it < n_it; ++it) {
        const int qs = it % kStages;
        if (!(ok = mbar_spin(bar(B_QDO_FULL + qs), (it / kStages) & 1, w))) break;
        if (!(ok = mbar_spin(bar(B_DP_FREE), (it & 1) ^ 1, w))) break;
        tc_fence_after();
        const uint32_t bq = sb + OFF_DO + qs * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_bf16(tmem + TM_DPT, sdesc_sw128(sb + OFF_V + off, 16, 1024), sdesc_sw128(bq + off, 16, 1024), id_s,
                    kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_DP_FULL));
      }
      umma_commit(bar(B_DRAIN_P));
      mbar_wait_drain(bar(B_DRAIN_P), 0, p.status);
    }
  } else if (warp == kGrad) {
    if (lane == 0) {
      // dV(i) += P^T(i) dO(i) half by half as each half's P^T is written
      // (then that half's S^T columns are free); dK(i) += dS^T(i) Q(i) once
      // dS^T is written (then the dP^T columns and the Q/dO stage are free:
      // S^T(i) and dP^T(i) had completed before the compute warps could write
      // P^T and dS^T).
      constexpr uint32_t id_g = idesc_bf16(128, 128, 0, 1);  // A from TMEM, B MN-major
      auto issue_grad = [&](int it, int tm_a, uint32_t b_base, int tm_d, int kk0, int kk1) {
        const uint32_t bq = b_base + (it % kStages) * kTile;
        for (int kk = kk0; kk < kk1; ++kk) {
          // queries 16 kk .. 16 kk + 15: compute group kk / 2 wrote them at
          // its own 32-column slice
          const uint32_t a = tmem + tm_a + (kk >> 1) * 32 + (kk & 1) * 8;
          umma_bf16_ts(tmem + tm_d, a, sdesc_sw128(bq + kk * 2048, kHalf, 1024), id_g,
                       (carry_in || it > 0 || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = true;
      if (carry_in) ok = mbar_wait(bar(B_CARRY_READY), 0, w);
      for (int it = 0; ok && it < n_it; ++it) {
        for (int hf = 0; hf < 2; ++hf) {
          if (!(ok = mbar_spin(bar(B_P_FULL + hf), it & 1, w))) break;
          tc_fence_after();
          issue_grad(it, TM_ST, sb + OFF_DO, TM_DV, 4 * hf, 4 * hf + 4);
          umma_commit(bar(B_S_FREE + hf));
        }
        if (!ok) break;
        if (!(ok = mbar_spin(bar(B_DS_FULL), it & 1, w))) break;
        tc_fence_after();
        issue_grad(it, TM_DPT, sb + OFF_Q, TM_DK, 0, 8);
        umma_commit(bar(B_DP_FREE));
        umma_commit(bar(B_QDO_EMPTY + it % kStages));
      }
      if (ok) umma_commit(bar(B_DKV_DONE));
      umma_commit(bar(B_DRAIN_G));
      mbar_wait_drain(bar(B_DRAIN_G), 0, p.status);
    }
  } else {
    // Compute warps: quadrant (warp & 3) of the key rows, group (warp >> 2)
    // of 32 query columns of each tile.
    const int quad = warp & 3;
    const int grp = warp >> 2;
    const int r = quad * 32 + lane;  // key row = TMEM lane
    const int kpos = kb * 128 + r;
    const bool valid = kpos < p.L;
    const uint32_t trow = tmem_lane_addr(tmem, quad, 0);
    const float sl2 = p.scale_log2;
    // Carry and epilogue: groups 0-1 own dK, 2-3 own dV, 64 columns each.
    const int which = grp >> 1;
    const int col0 = (grp & 1) * 64;
    float* my_carry = p.dkv_carry + (static_cast<int64_t>(kv * 2 + which) * p.L + kpos) * kHeadDim + col0;
    const uint32_t my_tm = trow + (which == 0 ? TM_DK : TM_DV) + col0;
    bool ok = true;
    if (carry_in) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 x = valid ? ld_global_nc_v4(my_carry + c * 32 + q * 4) : make_uint4(0, 0, 0, 0);
          v[4 * q] = x.x;
          v[4 * q + 1] = x.y;
          v[4 * q + 2] = x.z;
          v[4 * q + 3] = x.w;
        }
        tmem_st32(my_tm + c * 32, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_CARRY_READY));
    }
    const uint32_t ts = trow + TM_ST + grp * 32;
    const uint32_t td = trow + TM_DPT + grp * 32;
    for (int it = 0; it < n_it; ++it) {
      const int hl = kv * p.g_loc + it / nqt;
      const int qt = kb + it % nqt;
      const int q0 = qt * 128 + grp * 32;  // query of this warp's first column
      // Without its record (all 64 queries past L) the slice is all zero.
      const bool live = 2 * qt + (grp >> 1) < n_q64;
      // This warp's 32 queries in their record: -LSE*log2(e) at +0, Delta at
      // +64.  Lane c loads query c's pair now, ahead of the waits, and the
      // values reach the other lanes by shuffle.
      const float* rec = p.ld + (static_cast<int64_t>(hl) * n_q64 + 2 * qt + (grp >> 1)) * 128 + (grp & 1) * 32;
      const float nl = live ? __ldg(rec + lane) : 0.f;
      const float dl = live ? __ldg(rec + 64 + lane) : 0.f;
      // ---- phase 1: P^T over the S^T columns, 16 at a time; the packed
      // P^T of columns 16 h .. 16 h + 15 goes to columns 8 h .. 8 h + 7, which
      // this warp has already read.
      if (!(ok = warp_wait<false, true>(bar(B_S_FULL + (grp >> 1)), it & 1, w))) break;
      tc_fence_after();
      float pf[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t sv[16];
        tmem_ld16(ts + 16 * h, sv);
        tmem_ld_wait(sv);
        if (!live) {
#pragma unroll
          for (int c = 0; c < 16; ++c) pf[16 * h + c] = 0.f;
        } else if (qt == kb) {  // the diagonal tile (warp-uniform)
          p_slice<true>(sv, nl, 16 * h, sl2, q0, kpos, pf + 16 * h);
        } else {
          p_slice<false>(sv, nl, 16 * h, sl2, q0, kpos, pf + 16 * h);
        }
        uint32_t pk[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) pk[c] = pack_bf16x2(pf[16 * h + 2 * c], pf[16 * h + 2 * c + 1]);
        tmem_st8(ts + 8 * h, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P_FULL + (grp >> 1)));
      // ---- phase 2: dS^T = P^T * (dP^T - Delta) over the dP^T columns
      if (!(ok = warp_wait<false, true>(bar(B_DP_FULL), it & 1, w))) break;
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t dv[16];
        tmem_ld16(td + 16 * h, dv);
        tmem_ld_wait(dv);
        uint32_t dd[8];
        if (!live) {
#pragma unroll
          for (int c = 0; c < 8; ++c) dd[c] = 0u;
        } else {
          dst_slice(dv, pf + 16 * h, dl, 16 * h, dd);
        }
        tmem_st8(td + 8 * h, dd);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DS_FULL));
    }
    if (ok) ok = warp_wait<false, true>(bar(B_DKV_DONE), 0, w);
    if (ok) {
      tc_fence_after();
      if (p.carry_out) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          tmem_ld32(my_tm + c * 32, v);
          tmem_ld_wait(v);
          if (valid) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_global_v4(my_carry + c * 32 + q * 4, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
        }
      } else if (which == 0) {
        // dK: scale, rotate back by -angle (layer path), bf16 (+ residual).
        // This warp writes the RoPE pairs (i, i + 64), i in [32 (grp & 1), +32).
        __nv_bfloat16* outk = p.dk + static_cast<int64_t>(kpos) * p.dkv_row + static_cast<int64_t>(kv) * p.dkv_head;
        const float2* tab = p.rope ? p.rope + static_cast<int64_t>(kpos) * 64 : nullptr;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i0 = (grp & 1) * 32 + hh * 16;
          uint32_t a[16], b[16];
          tmem_ld16(trow + TM_DK + i0, a);
          tmem_ld16(trow + TM_DK + 64 + i0, b);
          tmem_ld_wait(a);
          tmem_ld_wait(b);
          float lo[16], hi[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float x0 = __uint_as_float(a[i]) * p.scale;
            const float x1 = __uint_as_float(b[i]) * p.scale;
            if (tab && valid) {
              const float2 cs = tab[i0 + i];
              lo[i] = x0 * cs.x + x1 * cs.y;
              hi[i] = x1 * cs.x - x0 * cs.y;
            } else {
              lo[i] = x0;
              hi[i] = x1;
            }
          }
          if (valid) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              store8_bf16_split(outk + i0 + q * 8, lo + 8 * q, p.lo_off);
              store8_bf16_split(outk + 64 + i0 + q * 8, hi + 8 * q, p.lo_off);
            }
          }
        }
      } else {
        __nv_bfloat16* outv =
            p.dv + static_cast<int64_t>(kpos) * p.dkv_row + static_cast<int64_t>(kv) * p.dkv_head + col0;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          tmem_ld32(my_tm + c * 32, v);
          tmem_ld_wait(v);
          if (valid) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
#pragma unroll
            for (int q = 0; q < 4; ++q) store8_bf16_split(outv + c * 32 + q * 8, f + 8 * q, p.lo_off);
          }
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == kMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_attn_bwd_dq(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& dO, const AttnBwdParams& p, int n_qblocks, cudaStream_t s) {
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dq::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(n_qblocks * p.nheads);
  attn_bwd_dq_kernel<<<grid, dq::kThreadsDq, dq::kSmemBytes, s>>>(q, k, v, dO, p);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dkdv(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& dO, const AttnBwdParams& p, int n_kblocks, cudaStream_t s) {
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(n_kblocks * p.nkv);
  attn_bwd_dkdv_kernel<<<grid, dkv::kThreadsKv, dkv::kSmemBytes, s>>>(q, k, v, dO, p);
  return cudaGetLastError();
}

}  // namespace upipe
