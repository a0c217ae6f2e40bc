// Exact causal attention forward for one head-chunk, tcgen05 + TMEM.
//
// What it computes: for query head h with KV head h / g, S = Q K^T / sqrt(d)
// with keys j <= i visible to query i, O = softmax(S) V and
// LSE_i = ln sum_j exp(S_ij).  The method keeps this formula unchanged and
// only changes which heads are resident at a time ("Untied Ulysses Pushes
// Llama-3-8B Training to 5 Million Tokens", paragraph on intermediate
// buffers: "not a new attention formula, but a different memory schedule").
//
// Design (sm_103a).  The tensor core reads shared-memory operands at about
// 128 B/clk per SM, which an M=128 product with both operands in shared
// memory saturates; so everything that can live in TMEM does:
//  * one CTA = one 128-query tile of one head, heaviest (most KV blocks)
//    first so the causal triangle balances across SMs;
//  * warp 4 streams Q once and K/V blocks of 128 keys through 3-stage TMA
//    rings (128-byte swizzle); the softmax warps copy Q into TMEM once;
//  * warp 5 issues S(j) = Q K^T (Q from TMEM) into the TMEM score buffer;
//    warp 6 issues O += P V (P from TMEM).  A thread issues a tcgen05.mma
//    only about every 100 cycles, hence two issuers;
//  * warps 0-3 own one query row per thread (the TMEM lane), so row max and
//    row sum are thread-local.  They write P as packed bf16 into one of two
//    TMEM buffers of its own: the score buffer is free again as soon as it
//    has been read (S(j + 1) overlaps the rest of the softmax of block j),
//    and P(j) need not wait for P V of block j - 1.  O is rescaled in TMEM
//    only when a row maximum grows by more than 2^8, which bounds every
//    exponent and keeps the result exact up to rounding.
//
// Three modes (a template parameter):
//  * kOnline: the online softmax above; writes O and LSE;
//  * kLseIn: the row's LSE is given (the forward's), so every block's
//    probabilities are final at once -- P = exp2(S log2(e)/sqrt(d) -
//    LSE log2(e)), the softmax's own definition -- and O = sum_j P_j V_j
//    needs no running maximum, rescaling, row sum or division.  The
//    backward's recomputation of O uses it: its P is the P the backward
//    kernels use, rounded to bf16 the same way;
//  * kLseOnly: row maximum and sum only (no P V, no O), for a forward that
//    keeps O for the backward and then writes it with kLseIn, so that a
//    kept O and a recomputed O are the same bits.
#include "sm103_ptx.cuh"

namespace upipe {
namespace {

constexpr int kTile = 128 * 128 * 2;  // [128][128] bf16, stored as two 64-column halves
constexpr int kHalf = kTile / 2;
constexpr int kStages = 3;            // K and V ring depth
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + kTile;
constexpr int OFF_V = OFF_K + kStages * kTile;
constexpr int OFF_BAR = OFF_V + kStages * kTile;

enum {
  B_Q_FULL,
  B_Q_TMEM,  // Q copied into TMEM by the softmax warps
  B_K_FULL,
  B_K_EMPTY = B_K_FULL + kStages,
  B_V_FULL = B_K_EMPTY + kStages,
  B_V_EMPTY = B_V_FULL + kStages,
  B_S_FULL = B_V_EMPTY + kStages,
  B_S_READ,                  // the softmax warps have read the score buffer
  B_P_FULL,                  // P written, per P buffer
  B_P_EMPTY = B_P_FULL + 2,  // P V done: that P buffer free, O up to date
  B_DRAIN = B_P_EMPTY + 2,
  B_DRAIN_PV,
  B_COUNT
};
constexpr int OFF_TMEM_SLOT = OFF_BAR + B_COUNT * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 8;
constexpr int kSmemBytes = OFF_ABORT + 8 + 1024;  // + alignment slack

constexpr int kThreads = 224;  // softmax warps 0-3, producer 4, S issuer 5, PV issuer 6
constexpr uint32_t kTmemCols = 512;
constexpr int TM_Q = 0;    // Q, packed bf16: columns [0, 64)
constexpr int TM_S = 64;   // scores: [64, 192)
constexpr int TM_O = 192;  // O accumulator: [192, 320)
constexpr int TM_P = 320;  // two P buffers, packed bf16: [320, 384), [384, 448)

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, const __grid_constant__ AttnFwdParams p) {
  constexpr bool kWithPV = MODE != kLseOnly;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Heads vary fastest: the CTAs in flight hold the same query blocks of
  // every head, whose K/V blocks (shared within a GQA group) stay in L2, and
  // the query blocks with the most KV blocks launch first.
  const int h = static_cast<int>(blockIdx.x) % p.nheads;
  const int qb = static_cast<int>(gridDim.x) / p.nheads - 1 - static_cast<int>(blockIdx.x) / p.nheads;
  const int kz = p.k_z0 + h / p.g_loc;
  const int vz = p.v_z0 + h / p.g_loc;
  const int n_kv = qb + 1;  // causal: KV blocks 0..qb
  auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  const WaitCtl w{abort_flag, p.status, p.limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    mbar_init(bar(B_Q_TMEM), 4);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_K_FULL + s), 1);
      mbar_init(bar(B_K_EMPTY + s), 1);
      mbar_init(bar(B_V_FULL + s), 1);
      mbar_init(bar(B_V_EMPTY + s), 1);
    }
    mbar_init(bar(B_S_FULL), 1);
    mbar_init(bar(B_S_READ), 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_P_FULL + b), 4);
      mbar_init(bar(B_P_EMPTY + b), 1);
    }
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN_PV), 1);
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&mq);
      tma_prefetch_map(&mk);
      tma_prefetch_map(&mv);
      mbar_expect_tx(bar(B_Q_FULL), kTile);
      tma_load_3d(sb + OFF_Q, &mq, bar(B_Q_FULL), 0, qb * 128, p.q_z0 + h);
      tma_load_3d(sb + OFF_Q + kHalf, &mq, bar(B_Q_FULL), 64, qb * 128, p.q_z0 + h);
      int last_k[kStages], last_v[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last_k[s] = last_v[s] = -1;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        if (!mbar_wait(bar(B_K_EMPTY + s), ph ^ 1, w)) break;
        mbar_expect_tx(bar(B_K_FULL + s), kTile);
        tma_load_3d(sb + OFF_K + s * kTile, &mk, bar(B_K_FULL + s), 0, j * 128, kz);
        tma_load_3d(sb + OFF_K + s * kTile + kHalf, &mk, bar(B_K_FULL + s), 64, j * 128, kz);
        last_k[s] = j;
        if constexpr (kWithPV) {
          if (!mbar_wait(bar(B_V_EMPTY + s), ph ^ 1, w)) break;
          mbar_expect_tx(bar(B_V_FULL + s), kTile);
          tma_load_3d(sb + OFF_V + s * kTile, &mv, bar(B_V_FULL + s), 0, j * 128, vz);
          tma_load_3d(sb + OFF_V + s * kTile + kHalf, &mv, bar(B_V_FULL + s), 64, j * 128, vz);
          last_v[s] = j;
        }
      }
      if (*abort_flag) {  // let every issued copy land before the CTA exits
        mbar_wait_drain(bar(B_Q_FULL), 0, p.status);
        for (int s = 0; s < kStages; ++s) {
          if (last_k[s] >= 0) mbar_wait_drain(bar(B_K_FULL + s), (last_k[s] / kStages) & 1, p.status);
          if (last_v[s] >= 0) mbar_wait_drain(bar(B_V_FULL + s), (last_v[s] / kStages) & 1, p.status);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);  // Q (TMEM) x K (smem, K-major)
      // S(j) once K(j) has landed and the softmax warps have read S(j - 1).
      bool ok = mbar_spin(bar(B_Q_TMEM), 0, w);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % kStages;
        if (!(ok = mbar_spin(bar(B_K_FULL + s), (j / kStages) & 1, w))) break;
        if (!(ok = mbar_spin(bar(B_S_READ), (j & 1) ^ 1, w))) break;
        tc_fence_after();
        const uint32_t ka = sb + OFF_K + s * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          umma_bf16_ts(tmem + TM_S, tmem + TM_Q + kk * 8,
                       sdesc_sw128(ka + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_S_FULL));
        umma_commit(bar(B_K_EMPTY + s));
      }
      umma_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0, p.status);
    }
  } else if (warp == 6) {
    // ----------------------------------------------------------- PV issuer
    if (kWithPV && lane == 0) {
      constexpr uint32_t id_o = idesc_bf16(128, 128, 0, 1);  // P (TMEM) x V (smem, MN-major)
      bool ok = true;
      for (int j = 0; ok && j < n_kv; ++j) {
        const int b = j & 1;
        const int s = j % kStages;
        if (!(ok = mbar_spin(bar(B_P_FULL + b), (j >> 1) & 1, w))) break;
        if (!(ok = mbar_spin(bar(B_V_FULL + s), (j / kStages) & 1, w))) break;
        tc_fence_after();
        const uint32_t va = sb + OFF_V + s * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          umma_bf16_ts(tmem + TM_O, tmem + TM_P + b * 64 + kk * 8, sdesc_sw128(va + kk * 2048, kHalf, 1024), id_o,
                       (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_P_EMPTY + b));
        umma_commit(bar(B_V_EMPTY + s));
      }
      umma_commit(bar(B_DRAIN_PV));
      mbar_wait_drain(bar(B_DRAIN_PV), 0, p.status);
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int r = warp * 32 + lane;  // query row in the tile = TMEM lane
    const int qpos = qb * 128 + r;
    const uint32_t trow = tmem_lane_addr(tmem, warp, 0);
    const float sl2 = p.scale_log2;
    float m_use = -INFINITY;  // running max used as the exponent offset (log2 domain)
    float l = 0.f;
    // kLseIn: -LSE * log2(e) of this row (0 past L: such rows are never stored).
    const float nl = MODE == kLseIn && qpos < p.L
                         ? -p.lse_in[static_cast<int64_t>(h) * p.L + qpos] * 1.4426950408889634074f
                         : 0.f;
    // Q row r -> TMEM (packed bf16, element pairs per column).
    bool ok = warp_wait(bar(B_Q_FULL), 0, w);
    if (ok) {
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {
        uint32_t q[32];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 v = ld_shared_v4(sb + OFF_Q + hq * kHalf + sw128_offset(r, ch));
          q[4 * ch] = v.x;
          q[4 * ch + 1] = v.y;
          q[4 * ch + 2] = v.z;
          q[4 * ch + 3] = v.w;
        }
        tmem_st32(trow + TM_Q + hq * 32, q);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_Q_TMEM));
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      const int b = j & 1;  // P buffer
      if (!(ok = warp_wait(bar(B_S_FULL), j & 1, w))) break;
      tc_fence_after();
      const uint32_t tsb = trow + TM_S;
      uint32_t v0[32], v1[32], v2[32], v3[32];
      tmem_ld32(tsb + 0, v0);
      tmem_ld32(tsb + 32, v1);
      tmem_ld32(tsb + 64, v2);
      tmem_ld32(tsb + 96, v3);
      tmem_ld_wait(v0);
      tmem_ld_wait(v1);
      tmem_ld_wait(v2);
      tmem_ld_wait(v3);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_S_READ));  // S(j + 1) may overwrite the scores

      float x[128];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        x[c] = __uint_as_float(v0[c]);
        x[32 + c] = __uint_as_float(v1[c]);
        x[64 + c] = __uint_as_float(v2[c]);
        x[96 + c] = __uint_as_float(v3[c]);
      }
      if (j == qb) {  // diagonal block: key c visible iff c <= r
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > r) x[c] = -INFINITY;
      }
      if constexpr (MODE == kLseIn) {
        // Final probabilities at once: P = exp2(S sl2 - LSE log2(e)).
        uint32_t pk0[32], pk1[32];
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const uint64_t nlx2 = f2_pack(nl, nl);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float t0, t1, t2, t3;
          f2_unpack(f2_fma(f2_pack(x[c], x[c + 1]), sl2x2, nlx2), t0, t1);
          f2_unpack(f2_fma(f2_pack(x[64 + c], x[64 + c + 1]), sl2x2, nlx2), t2, t3);
          pk0[c >> 1] = pack_bf16x2(ex2_approx(t0), ex2_approx(t1));
          pk1[c >> 1] = pack_bf16x2(ex2_approx(t2), ex2_approx(t3));
        }
        if (j >= 2) {
          if (!(ok = warp_wait(bar(B_P_EMPTY + b), ((j >> 1) & 1) ^ 1, w))) break;
          tc_fence_after();
        }
        tmem_st32(trow + TM_P + b * 64 + 0, pk0);
        tmem_st32(trow + TM_P + b * 64 + 32, pk1);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_P_FULL + b));
        continue;
      }
      // Row max: four independent chains of 3-input max.
      float mc[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
      for (int c = 4; c < 124; c += 8) {
        mc[0] = fmax3(mc[0], x[c], x[c + 1]);
        mc[1] = fmax3(mc[1], x[c + 2], x[c + 3]);
        mc[2] = fmax3(mc[2], x[c + 4], x[c + 5]);
        mc[3] = fmax3(mc[3], x[c + 6], x[c + 7]);
      }
      mc[0] = fmax3(mc[0], x[124], x[125]);
      mc[1] = fmax3(mc[1], x[126], x[127]);
      const float mx = fmaxf(fmax3(mc[0], mc[1], mc[2]), mc[3]);
      const float m_new = fmaxf(m_use, mx * sl2);
      const bool need = m_new > m_use + 8.0f;
      if (kWithPV && j > 0 && __any_sync(0xffffffffu, need)) {
        // O holds PV(0..j-1) once PV(j - 1) completes: rescale the rows
        // that moved.
        if (!(ok = warp_wait(bar(B_P_EMPTY + ((j - 1) & 1)), ((j - 1) >> 1) & 1, w))) break;
        tc_fence_after();
        const float f = need ? ex2_approx(m_use - m_new) : 1.f;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t o[32];
          tmem_ld32(trow + TM_O + c4 * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
          tmem_st32(trow + TM_O + c4 * 32, o);
        }
        l *= f;
      } else if (!kWithPV && need) {
        l *= ex2_approx(m_use - m_new);  // no O to rescale: only the row sum
      }
      if (need) m_use = m_new;

      uint32_t pk0[32], pk1[32];
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      const uint64_t nmx2 = f2_pack(-m_use, -m_use);
      uint64_t acc[4] = {0, 0, 0, 0};  // (+0, +0) pairs
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float t0, t1, t2, t3;
        f2_unpack(f2_fma(f2_pack(x[c], x[c + 1]), sl2x2, nmx2), t0, t1);
        f2_unpack(f2_fma(f2_pack(x[64 + c], x[64 + c + 1]), sl2x2, nmx2), t2, t3);
        const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
        const float p2 = ex2_approx(t2), p3 = ex2_approx(t3);
        acc[(c >> 1) & 1] = f2_add(acc[(c >> 1) & 1], f2_pack(p0, p1));
        acc[2 + ((c >> 1) & 1)] = f2_add(acc[2 + ((c >> 1) & 1)], f2_pack(p2, p3));
        pk0[c >> 1] = pack_bf16x2(p0, p1);
        pk1[c >> 1] = pack_bf16x2(p2, p3);
      }
      float rs = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a, b;
        f2_unpack(acc[i], a, b);
        rs += a + b;
      }
      l += rs;
      if constexpr (!kWithPV) continue;
      // P buffer b held P(j - 2) until PV(j - 2) completed.
      if (j >= 2) {
        if (!(ok = warp_wait(bar(B_P_EMPTY + b), ((j >> 1) & 1) ^ 1, w))) break;
        tc_fence_after();
      }
      tmem_st32(trow + TM_P + b * 64 + 0, pk0);
      tmem_st32(trow + TM_P + b * 64 + 32, pk1);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P_FULL + b));
    }
    // PV products complete in issue order: the last one completing means O is final.
    if (kWithPV && ok) ok = warp_wait(bar(B_P_EMPTY + ((n_kv - 1) & 1)), ((n_kv - 1) >> 1) & 1, w);
    if (ok && !kWithPV) {
      if (qpos < p.L) p.lse[static_cast<int64_t>(h) * p.L + qpos] = (m_use + log2f(l)) * 0.69314718055994530942f;
    } else if (ok) {
      tc_fence_after();
      const float inv = MODE == kLseIn ? 1.f : 1.f / l;
      const bool valid = qpos < p.L;
      __nv_bfloat16* orow = p.o + static_cast<int64_t>(qpos) * p.o_row + static_cast<int64_t>(h) * p.o_head;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t o[32];
        tmem_ld32(trow + TM_O + c4 * 32, o);
        tmem_ld_wait(o);
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            st_global_v4(orow + c4 * 32 + q * 8,
                         pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv),
                         pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv),
                         pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv),
                         pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv));
          }
        }
      }
      if (MODE == kOnline && valid && p.write_lse)
        p.lse[static_cast<int64_t>(h) * p.L + qpos] = (m_use + log2f(l)) * 0.69314718055994530942f;
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const AttnFwdParams& p,
                        int n_qblocks, cudaStream_t s) {
  cudaError_t e =
      cudaFuncSetAttribute(attn_fwd_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(n_qblocks * p.nheads);
  attn_fwd_kernel<MODE><<<grid, kThreads, kSmemBytes, s>>>(q, k, v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const AttnFwdParams& p, int n_qblocks, cudaStream_t s) {
  switch (p.mode) {
    case kOnline: return launch_mode<kOnline>(q, k, v, p, n_qblocks, s);
    case kLseIn: return launch_mode<kLseIn>(q, k, v, p, n_qblocks, s);
    case kLseOnly: return launch_mode<kLseOnly>(q, k, v, p, n_qblocks, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace upipe
