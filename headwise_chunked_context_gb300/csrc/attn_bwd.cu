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
//  * dq kernel: one CTA per (query head, 128-query tile) walks its KV blocks
//    in ascending order and accumulates dQ in TMEM;
//  * dkdv kernel: one CTA per (KV head, 128-key tile) walks the query heads
//    that read this KV head (ascending) and, for each, the 64-query tiles at
//    or after the key tile (ascending), accumulating dK and dV in TMEM.  When
//    a chunk holds fewer query heads than a KV group (U < g) the partial sums
//    are carried in fp32 between chunks and reloaded into TMEM, which keeps
//    the same order as a single pass over the whole group.
#include "sm103_ptx.cuh"

namespace upipe {
namespace {

constexpr float kLog2e = 1.4426950408889634074f;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, w));
}

// ============================================================== dQ kernel

namespace dq {
constexpr int kTile = 128 * 128 * 2;
constexpr int kHalf = kTile / 2;
constexpr int OFF_Q = 0;
constexpr int OFF_DO = OFF_Q + kTile;
constexpr int OFF_K = OFF_DO + kTile;     // 2 stages
constexpr int OFF_V = OFF_K + 2 * kTile;  // 2 stages
constexpr int OFF_DS = OFF_V + 2 * kTile;
constexpr int OFF_BAR = OFF_DS + kTile;
enum {
  B_QDO_FULL,
  B_K_FULL,
  B_K_EMPTY = B_K_FULL + 2,
  B_V_FULL = B_K_EMPTY + 2,
  B_V_EMPTY = B_V_FULL + 2,
  B_SDP_FULL = B_V_EMPTY + 2,
  B_SDP_EMPTY,
  B_DS_FULL,
  B_DS_EMPTY,
  B_DQ_DONE,
  B_DRAIN,
  B_COUNT
};
constexpr int OFF_TMEM_SLOT = OFF_BAR + B_COUNT * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 8;
constexpr int kSmemBytes = OFF_ABORT + 8 + 1024;
constexpr int TM_S = 0, TM_DP = 128, TM_DQ = 256;
}  // namespace dq

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                       const __grid_constant__ AttnBwdParams p) {
  using namespace dq;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qb = gridDim.x - 1 - blockIdx.x;
  const int h = blockIdx.y;
  const int kz = p.k_z0 + h / p.g_loc;
  const int vz = p.v_z0 + h / p.g_loc;
  const int n_kv = qb + 1;
  auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  const WaitCtl w{abort_flag, p.status, p.limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QDO_FULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_K_FULL + s), 1);
      mbar_init(bar(B_K_EMPTY + s), 1);
      mbar_init(bar(B_V_FULL + s), 1);
      mbar_init(bar(B_V_EMPTY + s), 1);
    }
    mbar_init(bar(B_SDP_FULL), 1);
    mbar_init(bar(B_SDP_EMPTY), 4);
    mbar_init(bar(B_DS_FULL), 4);
    mbar_init(bar(B_DS_EMPTY), 1);
    mbar_init(bar(B_DQ_DONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(sb + OFF_TMEM_SLOT, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);

  if (warp == 4) {
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
      int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
      for (int j = 0; j < n_kv; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(bar(B_K_EMPTY + s), ph ^ 1, w)) break;
        mbar_expect_tx(bar(B_K_FULL + s), kTile);
        tma_load_3d(sb + OFF_K + s * kTile, &mk, bar(B_K_FULL + s), 0, j * 128, kz);
        tma_load_3d(sb + OFF_K + s * kTile + kHalf, &mk, bar(B_K_FULL + s), 64, j * 128, kz);
        last_k[s] = j;
        if (!mbar_wait(bar(B_V_EMPTY + s), ph ^ 1, w)) break;
        mbar_expect_tx(bar(B_V_FULL + s), kTile);
        tma_load_3d(sb + OFF_V + s * kTile, &mv, bar(B_V_FULL + s), 0, j * 128, vz);
        tma_load_3d(sb + OFF_V + s * kTile + kHalf, &mv, bar(B_V_FULL + s), 64, j * 128, vz);
        last_v[s] = j;
      }
      if (*abort_flag) {
        mbar_wait_drain(bar(B_QDO_FULL), 0, p.status);
        for (int s = 0; s < 2; ++s) {
          if (last_k[s] >= 0) mbar_wait_drain(bar(B_K_FULL + s), (last_k[s] >> 1) & 1, p.status);
          if (last_v[s] >= 0) mbar_wait_drain(bar(B_V_FULL + s), (last_v[s] >> 1) & 1, p.status);
        }
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_bf16(128, 128, 0, 0);  // S = Q K^T, dP = dO V^T
      constexpr uint32_t id_kn = idesc_bf16(128, 128, 0, 1);  // dQ += dS K (K as MN-major B)
      auto issue_dq = [&](int jj) -> bool {
        const int s = jj & 1;
        if (!mbar_wait(bar(B_DS_FULL), jj & 1, w)) return false;
        tc_fence_after();
        const uint32_t ka = sb + OFF_K + s * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          umma_bf16(tmem + TM_DQ, sdesc_sw128(sb + OFF_DS + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024),
                    sdesc_sw128(ka + kk * 2048, kHalf, 1024), id_kn, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_DS_EMPTY));
        umma_commit(bar(B_K_EMPTY + s));
        return true;
      };
      bool ok = mbar_wait(bar(B_QDO_FULL), 0, w);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!(ok = mbar_wait(bar(B_K_FULL + s), ph, w))) break;
        if (!(ok = mbar_wait(bar(B_V_FULL + s), ph, w))) break;
        if (!(ok = mbar_wait(bar(B_SDP_EMPTY), (j & 1) ^ 1, w))) break;
        tc_fence_after();
        const uint32_t ka = sb + OFF_K + s * kTile;
        const uint32_t va = sb + OFF_V + s * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_bf16(tmem + TM_S, sdesc_sw128(sb + OFF_Q + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), id_kk,
                    kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_bf16(tmem + TM_DP, sdesc_sw128(sb + OFF_DO + off, 16, 1024), sdesc_sw128(va + off, 16, 1024), id_kk,
                    kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_SDP_FULL));
        umma_commit(bar(B_V_EMPTY + s));
        if (j >= 1) ok = issue_dq(j - 1);
      }
      if (ok && issue_dq(n_kv - 1)) umma_commit(bar(B_DQ_DONE));
      umma_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0, p.status);
    }
  } else {
    const int r = warp * 32 + lane;
    const int qpos = qb * 128 + r;
    const bool valid = qpos < p.L;
    const uint32_t trow = tmem_lane_addr(tmem, warp, 0);
    const float sl2 = p.scale_log2;
    const float lse2 = valid ? p.lse[static_cast<int64_t>(h) * p.L + qpos] * kLog2e : 0.f;
    const float dlt = valid ? p.delta[static_cast<int64_t>(h) * p.L + qpos] : 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!(ok = warp_wait(bar(B_SDP_FULL), j & 1, w))) break;
      if (!(ok = warp_wait(bar(B_DS_EMPTY), (j & 1) ^ 1, w))) break;
      tc_fence_after();
      const bool diag = (j == qb);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t s0[32], s1[32], d0[32], d1[32];
        tmem_ld32(trow + TM_S + half * 64, s0);
        tmem_ld32(trow + TM_S + half * 64 + 32, s1);
        tmem_ld32(trow + TM_DP + half * 64, d0);
        tmem_ld32(trow + TM_DP + half * 64 + 32, d1);
        tmem_ld_wait(s0);
        tmem_ld_wait(s1);
        tmem_ld_wait(d0);
        tmem_ld_wait(d1);
        if (half == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_SDP_EMPTY));
        }
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float ds2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int cc = c + e;
            const float sv = __uint_as_float(cc < 32 ? s0[cc] : s1[cc - 32]);
            const float dp = __uint_as_float(cc < 32 ? d0[cc] : d1[cc - 32]);
            float pv = ex2_approx(fmaf(sv, sl2, -lse2));
            if (diag && (half * 64 + cc) > r) pv = 0.f;
            ds2[e] = pv * (dp - dlt);
          }
          pk[c >> 1] = pack_bf16x2(ds2[0], ds2[1]);
        }
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          st_shared_v4(sb + OFF_DS + half * kHalf + sw128_offset(r, ch), pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2],
                       pk[4 * ch + 3]);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DS_FULL));
    }
    if (ok) ok = warp_wait(bar(B_DQ_DONE), 0, w);
    if (ok) {
      tc_fence_after();
      __nv_bfloat16* out = p.dq + static_cast<int64_t>(qpos) * p.dq_row + static_cast<int64_t>(h) * p.dq_head;
      const float2* tab = p.rope ? p.rope + static_cast<int64_t>(qpos) * 64 : nullptr;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
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
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ============================================================ dK/dV kernel

namespace dkv {
constexpr int kKV = 128 * 128 * 2;  // K or V tile: [128 keys][128 d]
constexpr int kKVHalf = kKV / 2;
constexpr int kQ = 64 * 128 * 2;    // Q or dO tile: [64 queries][128 d]
constexpr int kQHalf = kQ / 2;
constexpr int kPT = 128 * 64 * 2;   // P^T or dS^T tile: [128 keys][64 queries]
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + kKV;
constexpr int OFF_Q = OFF_V + kKV;     // 2 stages
constexpr int OFF_DO = OFF_Q + 2 * kQ;  // 2 stages
constexpr int OFF_PT = OFF_DO + 2 * kQ;  // 2 buffers
constexpr int OFF_DST = OFF_PT + 2 * kPT;  // 2 buffers
constexpr int OFF_LD = OFF_DST + 2 * kPT;  // 2 x (64 lse + 64 delta) floats
constexpr int OFF_BAR = OFF_LD + 2 * 512;
enum {
  B_KV_FULL,
  B_QDO_FULL,
  B_QDO_EMPTY = B_QDO_FULL + 2,
  B_SDP_FULL = B_QDO_EMPTY + 2,
  B_SDP_EMPTY = B_SDP_FULL + 2,
  B_PDS_FULL = B_SDP_EMPTY + 2,
  B_PDS_EMPTY = B_PDS_FULL + 2,
  B_LD_READY = B_PDS_EMPTY + 2,
  B_CARRY_READY = B_LD_READY + 2,
  B_DKV_DONE,
  B_DRAIN,
  B_COUNT
};
constexpr int OFF_TMEM_SLOT = OFF_BAR + B_COUNT * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 8;
constexpr int kSmemBytes = OFF_ABORT + 8 + 1024;
constexpr int TM_ST = 0, TM_DPT = 128, TM_DV = 256, TM_DK = 384;
}  // namespace dkv

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                         const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                         const __grid_constant__ AttnBwdParams p) {
  using namespace dkv;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kb = gridDim.x - 1 - blockIdx.x;  // key tiles near the start see the most queries
  const int kv = blockIdx.y;
  const int n_q64 = (p.L + 63) / 64;
  const int nqi = n_q64 - 2 * kb;  // query tiles at or after this key tile
  const int n_it = p.g_loc * nqi;
  auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  const WaitCtl w{abort_flag, p.status, p.limit_ns};
  const bool carry_in = p.carry_in != 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_KV_FULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QDO_FULL + s), 1);
      mbar_init(bar(B_QDO_EMPTY + s), 1);
      mbar_init(bar(B_SDP_FULL + s), 1);
      mbar_init(bar(B_SDP_EMPTY + s), 4);
      mbar_init(bar(B_PDS_FULL + s), 4);
      mbar_init(bar(B_PDS_EMPTY + s), 1);
      mbar_init(bar(B_LD_READY + s), 128);
    }
    mbar_init(bar(B_CARRY_READY), 4);
    mbar_init(bar(B_DKV_DONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(sb + OFF_TMEM_SLOT, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);

  if (warp == 4) {
    if (lane == 0) {
      tma_prefetch_map(&mq);
      tma_prefetch_map(&mk);
      tma_prefetch_map(&mv);
      tma_prefetch_map(&mdo);
      mbar_expect_tx(bar(B_KV_FULL), 2 * kKV);
      tma_load_3d(sb + OFF_K, &mk, bar(B_KV_FULL), 0, kb * 128, p.k_z0 + kv);
      tma_load_3d(sb + OFF_K + kKVHalf, &mk, bar(B_KV_FULL), 64, kb * 128, p.k_z0 + kv);
      tma_load_3d(sb + OFF_V, &mv, bar(B_KV_FULL), 0, kb * 128, p.v_z0 + kv);
      tma_load_3d(sb + OFF_V + kKVHalf, &mv, bar(B_KV_FULL), 64, kb * 128, p.v_z0 + kv);
      int last[2] = {-1, -1};
      for (int it = 0; it < n_it; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        const int hl = kv * p.g_loc + it / nqi;
        const int qi = 2 * kb + it % nqi;
        if (!mbar_wait(bar(B_QDO_EMPTY + s), ph ^ 1, w)) break;
        mbar_expect_tx(bar(B_QDO_FULL + s), 2 * kQ);
        tma_load_3d(sb + OFF_Q + s * kQ, &mq, bar(B_QDO_FULL + s), 0, qi * 64, p.q_z0 + hl);
        tma_load_3d(sb + OFF_Q + s * kQ + kQHalf, &mq, bar(B_QDO_FULL + s), 64, qi * 64, p.q_z0 + hl);
        tma_load_3d(sb + OFF_DO + s * kQ, &mdo, bar(B_QDO_FULL + s), 0, qi * 64, p.do_z0 + hl);
        tma_load_3d(sb + OFF_DO + s * kQ + kQHalf, &mdo, bar(B_QDO_FULL + s), 64, qi * 64, p.do_z0 + hl);
        last[s] = it;
      }
      if (*abort_flag) {
        mbar_wait_drain(bar(B_KV_FULL), 0, p.status);
        for (int s = 0; s < 2; ++s)
          if (last[s] >= 0) mbar_wait_drain(bar(B_QDO_FULL + s), (last[s] >> 1) & 1, p.status);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 64, 0, 0);   // S^T = K Q^T, dP^T = V dO^T
      constexpr uint32_t id_g = idesc_bf16(128, 128, 0, 1);  // dV += P^T dO, dK += dS^T Q
      auto issue_grad = [&](int ii) -> bool {
        const int s = ii & 1;
        const uint32_t ph = (ii >> 1) & 1;
        if (!mbar_wait(bar(B_PDS_FULL + s), ph, w)) return false;
        tc_fence_after();
        const uint32_t pt = sb + OFF_PT + s * kPT;
        const uint32_t dst = sb + OFF_DST + s * kPT;
        const uint32_t qa = sb + OFF_Q + s * kQ;
        const uint32_t da = sb + OFF_DO + s * kQ;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          umma_bf16(tmem + TM_DV, sdesc_sw128(pt + kk * 32, 16, 1024), sdesc_sw128(da + kk * 2048, kQHalf, 1024),
                    id_g, (carry_in || ii > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          umma_bf16(tmem + TM_DK, sdesc_sw128(dst + kk * 32, 16, 1024), sdesc_sw128(qa + kk * 2048, kQHalf, 1024),
                    id_g, (carry_in || ii > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_PDS_EMPTY + s));
        umma_commit(bar(B_QDO_EMPTY + s));
        return true;
      };
      bool ok = mbar_wait(bar(B_KV_FULL), 0, w);
      if (ok && carry_in) ok = mbar_wait(bar(B_CARRY_READY), 0, w);
      for (int it = 0; ok && it < n_it; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!(ok = mbar_wait(bar(B_QDO_FULL + s), ph, w))) break;
        if (!(ok = mbar_wait(bar(B_SDP_EMPTY + s), ph ^ 1, w))) break;
        tc_fence_after();
        const uint32_t qa = sb + OFF_Q + s * kQ;
        const uint32_t da = sb + OFF_DO + s * kQ;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t ko = (kk >> 2) * kKVHalf + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * kQHalf + (kk & 3) * 32;
          umma_bf16(tmem + TM_ST + s * 64, sdesc_sw128(sb + OFF_K + ko, 16, 1024), sdesc_sw128(qa + qo, 16, 1024),
                    id_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t ko = (kk >> 2) * kKVHalf + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * kQHalf + (kk & 3) * 32;
          umma_bf16(tmem + TM_DPT + s * 64, sdesc_sw128(sb + OFF_V + ko, 16, 1024), sdesc_sw128(da + qo, 16, 1024),
                    id_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_SDP_FULL + s));
        if (it >= 1) ok = issue_grad(it - 1);
      }
      if (ok && issue_grad(n_it - 1)) umma_commit(bar(B_DKV_DONE));
      umma_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0, p.status);
    }
  } else {
    const int r = warp * 32 + lane;  // key row = TMEM lane
    const int kpos = kb * 128 + r;
    const bool valid = kpos < p.L;
    const uint32_t trow = tmem_lane_addr(tmem, warp, 0);
    const float sl2 = p.scale_log2;
    float* carry_k = p.dkv_carry + (static_cast<int64_t>(kv * 2 + 0) * p.L + kpos) * kHeadDim;
    float* carry_v = p.dkv_carry + (static_cast<int64_t>(kv * 2 + 1) * p.L + kpos) * kHeadDim;
    bool ok = true;
    if (carry_in) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float* src = t == 0 ? carry_k : carry_v;
        const int col = t == 0 ? TM_DK : TM_DV;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 x = valid ? ld_global_nc_v4(src + c4 * 32 + q * 4) : make_uint4(0, 0, 0, 0);
            v[4 * q] = x.x;
            v[4 * q + 1] = x.y;
            v[4 * q + 2] = x.z;
            v[4 * q + 3] = x.w;
          }
          tmem_st32(trow + col + c4 * 32, v);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_CARRY_READY));
    }
    float* ld_smem = reinterpret_cast<float*>(smem + OFF_LD);
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      const int hl = kv * p.g_loc + it / nqi;
      const int qi = 2 * kb + it % nqi;
      {  // this query tile's LSE (log2 domain) and Delta into shared memory
        const int c = threadIdx.x & 63;
        const int q = qi * 64 + c;
        float val;
        if (threadIdx.x < 64)
          val = q < p.L ? p.lse[static_cast<int64_t>(hl) * p.L + q] * kLog2e : INFINITY;
        else
          val = q < p.L ? p.delta[static_cast<int64_t>(hl) * p.L + q] : 0.f;
        ld_smem[s * 128 + threadIdx.x] = val;
        mbar_arrive(bar(B_LD_READY + s));
      }
      if (!(ok = warp_wait(bar(B_LD_READY + s), ph, w))) break;
      if (!(ok = warp_wait(bar(B_SDP_FULL + s), ph, w))) break;
      tc_fence_after();
      uint32_t s0[32], s1[32], d0[32], d1[32];
      tmem_ld32(trow + TM_ST + s * 64, s0);
      tmem_ld32(trow + TM_ST + s * 64 + 32, s1);
      tmem_ld32(trow + TM_DPT + s * 64, d0);
      tmem_ld32(trow + TM_DPT + s * 64 + 32, d1);
      tmem_ld_wait(s0);
      tmem_ld_wait(s1);
      tmem_ld_wait(d0);
      tmem_ld_wait(d1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SDP_EMPTY + s));

      const float* lse_s = ld_smem + s * 128;
      const float* dl_s = lse_s + 64;
      const bool near_diag = qi * 64 < kb * 128 + 128;
      uint32_t pp[32], dd[32];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float pv2[2], ds2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int cc = c + e;
          const float sv = __uint_as_float(cc < 32 ? s0[cc] : s1[cc - 32]);
          const float dp = __uint_as_float(cc < 32 ? d0[cc] : d1[cc - 32]);
          float pv = ex2_approx(fmaf(sv, sl2, -lse_s[cc]));
          if (near_diag && qi * 64 + cc < kpos) pv = 0.f;
          pv2[e] = pv;
          ds2[e] = pv * (dp - dl_s[cc]);
        }
        pp[c >> 1] = pack_bf16x2(pv2[0], pv2[1]);
        dd[c >> 1] = pack_bf16x2(ds2[0], ds2[1]);
      }
      if (!(ok = warp_wait(bar(B_PDS_EMPTY + s), ph ^ 1, w))) break;
      const uint32_t pt = sb + OFF_PT + s * kPT;
      const uint32_t dst = sb + OFF_DST + s * kPT;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        st_shared_v4(pt + sw128_offset(r, ch), pp[4 * ch], pp[4 * ch + 1], pp[4 * ch + 2], pp[4 * ch + 3]);
        st_shared_v4(dst + sw128_offset(r, ch), dd[4 * ch], dd[4 * ch + 1], dd[4 * ch + 2], dd[4 * ch + 3]);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PDS_FULL + s));
    }
    if (ok) ok = warp_wait(bar(B_DKV_DONE), 0, w);
    if (ok) {
      tc_fence_after();
      if (p.carry_out) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          float* dstp = t == 0 ? carry_k : carry_v;
          const int col = t == 0 ? TM_DK : TM_DV;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t v[32];
            tmem_ld32(trow + col + c4 * 32, v);
            tmem_ld_wait(v);
            if (valid) {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                st_global_v4(dstp + c4 * 32 + q * 4, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
          }
        }
      } else {
        // dK: scale, rotate back by -angle (layer path), bf16.
        __nv_bfloat16* outk = p.dk + static_cast<int64_t>(kpos) * p.dkv_row + static_cast<int64_t>(kv) * p.dkv_head;
        __nv_bfloat16* outv = p.dv + static_cast<int64_t>(kpos) * p.dkv_row + static_cast<int64_t>(kv) * p.dkv_head;
        const float2* tab = p.rope ? p.rope + static_cast<int64_t>(kpos) * 64 : nullptr;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t a[32], b[32];
          tmem_ld32(trow + TM_DK + half * 32, a);
          tmem_ld32(trow + TM_DK + 64 + half * 32, b);
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
              store8_bf16_split(outk + half * 32 + q * 8, lo + 8 * q, p.lo_off);
              store8_bf16_split(outk + 64 + half * 32 + q * 8, hi + 8 * q, p.lo_off);
            }
          }
        }
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(trow + TM_DV + c4 * 32, v);
          tmem_ld_wait(v);
          if (valid) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
#pragma unroll
            for (int q = 0; q < 4; ++q) store8_bf16_split(outv + c4 * 32 + q * 8, f + 8 * q, p.lo_off);
          }
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 5) {
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
  dim3 grid(n_qblocks, p.nheads);
  attn_bwd_dq_kernel<<<grid, kThreads, dq::kSmemBytes, s>>>(q, k, v, dO, p);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dkdv(const CUtensorMap& q64, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& dO64, const AttnBwdParams& p, int n_kblocks, cudaStream_t s) {
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(n_kblocks, p.nkv);
  attn_bwd_dkdv_kernel<<<grid, kThreads, dkv::kSmemBytes, s>>>(q64, k, v, dO64, p);
  return cudaGetLastError();
}

}  // namespace upipe
