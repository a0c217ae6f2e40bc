// Memory-bound helpers: the RoPE cos/sin table, the Delta row sums of the
// attention backward, and the bounded-wait self-test.
#include "sm103_ptx.cuh"

namespace upipe {
namespace {

// RoPE angles p * theta^(-2i/d) (RoFormer, listed under "Builds on" on the
// "Untied Ulysses: Memory-Efficient Context Parallelism via Headwise
// Chunking" index page).  At p ~ 2^21 an fp32 product p * inv_freq is off by
// up to ~0.06 rad, so the angle is formed in fp64 and reduced modulo 2*pi in
// fp64 with a two-constant (Cody-Waite) split of 2*pi; only the reduced
// angle, |r| <= pi, goes through single-precision sincosf.
struct RopeFreqs {
  double inv_freq[64];
};

__global__ void rope_table_kernel(float2* __restrict__ table, int64_t L, const __grid_constant__ RopeFreqs f) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= L * 64) return;
  const int64_t pos = idx >> 6;
  const int i = static_cast<int>(idx & 63);
  const double a = static_cast<double>(pos) * f.inv_freq[i];
  constexpr double kTwoPiHi = 6.283185307179586232;       // nearest double to 2*pi
  constexpr double kTwoPiLo = 2.4492935982947064e-16;     // 2*pi - kTwoPiHi
  constexpr double kInvTwoPi = 0.15915494309189533577;
  const double k = rint(a * kInvTwoPi);
  double r = fma(-k, kTwoPiHi, a);
  r = fma(-k, kTwoPiLo, r);
  float s, c;
  sincosf(static_cast<float>(r), &s, &c);
  table[idx] = make_float2(c, s);
}

// LSE/Delta records for the core backward entry: for head h and row p,
// Delta = sum_k dO[p, h, k] * O[p, h, k] and -LSE * log2(e), stored per
// 64-row tile as [64 -LSE*log2(e) | 64 Delta]; rows past L get -inf / 0.
// 16 lanes per (row, head): each lane reads 16 bytes of O and of dO.
__global__ void delta_kernel(const __nv_bfloat16* __restrict__ o, int64_t o_row, int64_t o_head,
                             const __nv_bfloat16* __restrict__ dO, int64_t do_row, int64_t do_head,
                             const float* __restrict__ lse, float* __restrict__ ld, int64_t L, int nheads) {
  const int64_t n_q64 = (L + 63) / 64;
  const int64_t rows = n_q64 * 64;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t item = gid >> 4;  // (head, row)
  const int sub = threadIdx.x & 15;
  const bool live = item < rows * nheads;
  const int64_t hh = live ? item / rows : 0;
  const int64_t row = live ? item % rows : 0;
  const bool in = live && row < L;
  float acc = 0.f;
  if (in) {
    const uint4 a = ld_global_nc_v4(o + row * o_row + hh * o_head + sub * 8);
    const uint4 b = ld_global_nc_v4(dO + row * do_row + hh * do_head + sub * 8);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(bf16_lo(av[e]), bf16_lo(bv[e]), acc);
      acc = fmaf(bf16_hi(av[e]), bf16_hi(bv[e]), acc);
    }
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (live && sub == 0) {
    float* rec = ld + (hh * n_q64 + (row >> 6)) * 128;
    rec[row & 63] = in ? -lse[hh * L + row] * 1.4426950408889634074f : -INFINITY;
    rec[64 + (row & 63)] = in ? acc : 0.f;
  }
}

// One thread waits on an mbarrier that nothing arrives on.  The bounded wait
// runs out after `limit_ns` and records UPIPE_STATUS_TIMEOUT.
__global__ void wait_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl w{&abort_flag, status, limit_ns};
    mbar_wait(smem_u32(&bar), 0, w);
  }
}

struct ZeroRows {
  float* base;
  int64_t ld;
  int cols;
  int16_t blocks[kMaxSlots];
};

// One CTA per row: row (blockIdx.x & 127) of listed block blockIdx.x >> 7.
__global__ void __launch_bounds__(256) zero_rows_kernel(const __grid_constant__ ZeroRows z) {
  const int row = static_cast<int>(blockIdx.x);
  float4* dst = reinterpret_cast<float4*>(z.base + (static_cast<int64_t>(z.blocks[row >> 7]) * 128 + (row & 127)) * z.ld);
  for (int i = threadIdx.x; i < z.cols / 4; i += blockDim.x) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace

cudaError_t launch_zero_rows(float* base, int64_t ld, int cols, const int16_t* blocks, int n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (n > kMaxSlots || cols % 4 != 0 || ld % 4 != 0) return cudaErrorInvalidValue;
  ZeroRows z = {};
  z.base = base;
  z.ld = ld;
  z.cols = cols;
  for (int i = 0; i < n; ++i) z.blocks[i] = blocks[i];
  zero_rows_kernel<<<static_cast<unsigned>(n * 128), 256, 0, s>>>(z);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float2* table, int64_t L, double theta, cudaStream_t s) {
  RopeFreqs f;
  for (int i = 0; i < 64; ++i) f.inv_freq[i] = pow(theta, -2.0 * i / 128.0);
  const int64_t n = L * 64;
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  rope_table_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(table, L, f);
  return cudaGetLastError();
}

cudaError_t launch_delta(const __nv_bfloat16* o, int64_t o_row, int64_t o_head, const __nv_bfloat16* dO,
                         int64_t do_row, int64_t do_head, const float* lse, float* ld, int64_t L, int nheads,
                         cudaStream_t s) {
  const int64_t threads_total = (L + 63) / 64 * 64 * nheads * 16;
  const int threads = 256;
  const int64_t blocks = (threads_total + threads - 1) / threads;
  delta_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(o, o_row, o_head, dO, do_row, do_head, lse, ld,
                                                                  L, nheads);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace upipe
