// Sequence-tiled SwiGLU MLP and LM-head cross-entropy around the attention
// layer ("Untied Ulysses Pushes Llama-3-8B Training to 5 Million Tokens",
// talk write-up, paragraph on Arctic Long Sequence Training: MLPs and loss
// computations need no buffer spanning the whole sequence; they are chunked
// along the sequence axis).  Each entry point walks the sequence in tiles of
// T rows and reuses one workspace of T-row intermediates; every contraction
// runs on the tcgen05 GEMM kernel (gemm.cu), the softmax rows of the loss on
// the row kernel below.
//
// Weight gradients are carried in place across tiles: each tile's GEMM
// loads the fp32 partial into TMEM before its first product and adds its
// tokens' K blocks in ascending order, so every tile size that is a multiple
// of 64 performs the same fp32 additions in the same order as one tile of
// the whole sequence (identical bits).
#include <cmath>

#include "host.h"
#include "sm103_ptx.cuh"

namespace upipe {
namespace {

// ------------------------------------------------------------ loss rows

constexpr int kCeThreads = 512;

// One CTA per row: pass 1 forms the row's maximum and sum of exponentials
// (per thread with rescaling, then across the CTA), pass 2 writes
// dz = scale (exp(z - LSE) - [j == label]) as bf16.
__global__ void __launch_bounds__(kCeThreads) ce_rows_kernel(const float* __restrict__ z, int64_t ld_z, int V,
                                                             const int32_t* __restrict__ labels, float scale,
                                                             float* __restrict__ loss,
                                                             __nv_bfloat16* __restrict__ dz, int64_t ld_dz) {
  const int64_t row = blockIdx.x;
  const float* zr = z + row * ld_z;
  __nv_bfloat16* dr = dz + row * ld_dz;
  const int label = labels[row];
  const int n4 = V / 4;
  const float4* z4 = reinterpret_cast<const float4*>(zr);
  if (label < 0 || label >= V) {  // ignored token (negative) or a label outside the vocabulary (NaN loss)
    for (int i = threadIdx.x; i < n4; i += kCeThreads)
      *reinterpret_cast<uint2*>(dr + 4 * i) = make_uint2(0u, 0u);
    if (threadIdx.x == 0) loss[row] = label < 0 ? 0.f : __int_as_float(0x7fc00000);
    return;
  }
  float m = -INFINITY, s = 0.f;
  for (int i = threadIdx.x; i < n4; i += kCeThreads) {
    const float4 v = z4[i];
    const float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    if (mx > m) {
      s *= __expf(m - mx);
      m = mx;
    }
    s += __expf(v.x - m) + __expf(v.y - m) + __expf(v.z - m) + __expf(v.w - m);
  }
  // Combine (m, s) pairs: warp shuffles, then one value per warp.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float mn = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * __expf(m - mn)) + (m2 == -INFINITY ? 0.f : s2 * __expf(m2 - mn));
    m = mn;
  }
  __shared__ float sm[kCeThreads / 32], ss[kCeThreads / 32];
  __shared__ float s_lse;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sm[warp] = m;
    ss[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int w = 0; w < kCeThreads / 32; ++w) M = fmaxf(M, sm[w]);
    float S = 0.f;
    for (int w = 0; w < kCeThreads / 32; ++w)
      if (sm[w] != -INFINITY) S += ss[w] * __expf(sm[w] - M);
    const float lse = M + logf(S);
    s_lse = lse;
    loss[row] = lse - zr[label];
  }
  __syncthreads();
  const float lse = s_lse;
  for (int i = threadIdx.x; i < n4; i += kCeThreads) {
    const float4 v = z4[i];
    float p[4] = {__expf(v.x - lse), __expf(v.y - lse), __expf(v.z - lse), __expf(v.w - lse)};
    const int j0 = 4 * i;
    if (label >= j0 && label < j0 + 4) p[label - j0] -= 1.f;
    *reinterpret_cast<uint2*>(dr + j0) =
        make_uint2(pack_bf16x2(scale * p[0], scale * p[1]), pack_bf16x2(scale * p[2], scale * p[3]));
  }
}

// ------------------------------------------------------------ plans

struct MlpShape {
  int64_t L;
  int D, F, T;
};

bool check_mlp(const upipe_mlp_cfg* c, MlpShape* s) {
  if (!c || c->L < 1 || c->L > 0x7fffffffLL) return false;
  if (c->D < 128 || c->D % 128 || c->F < 128 || c->F % 128) return false;
  if (c->T < 128 || c->T % 128) return false;
  *s = MlpShape{c->L, c->D, c->F, c->T};
  return true;
}

struct CeShape {
  int64_t L;
  int D, V, T;
};

bool check_ce(const upipe_ce_cfg* c, CeShape* s) {
  if (!c || c->L < 1 || c->L > 0x7fffffffLL) return false;
  if (c->D < 128 || c->D % 128 || c->V < 128 || c->V % 128) return false;
  if (c->T < 128 || c->T % 128) return false;
  *s = CeShape{c->L, c->D, c->V, c->T};
  return true;
}

size_t al(size_t b) { return (b + 1023) / 1024 * 1024; }

// MLP workspace: H [T, F]; the backward adds dH [T, F] and [dG | dU] [T, 2F]
// (bf16).  Offsets: H, dH, dGU.
struct MlpPlan {
  size_t off_h = 0, off_dh = 0, off_dgu = 0, total = 0;
};
MlpPlan mlp_plan(const MlpShape& s, int pass) {
  MlpPlan p;
  const size_t tf = static_cast<size_t>(s.T) * s.F * 2;
  p.off_h = 0;
  size_t off = al(tf);
  if (pass == 1) {
    p.off_dh = off;
    off += al(tf);
    p.off_dgu = off;
    off += al(2 * tf);
  }
  p.total = off;
  return p;
}

// Loss workspace: the logits Z [T, V] fp32, then dZ [T, V] bf16.
size_t ce_z_bytes(const CeShape& s) { return al(static_cast<size_t>(s.T) * s.V * 4); }
size_t ce_total(const CeShape& s) { return ce_z_bytes(s) + al(static_cast<size_t>(s.T) * s.V * 2); }

using bf16 = __nv_bfloat16;

// C = A B^T with both operands K-major, through GK_OPROJ without a carry:
// bf16 `out` (leading dimension ld_out) or, with out == nullptr, fp32 into
// `f32` [M, N].
int gemm_abt(const CUtensorMap& ma, const CUtensorMap& mb, int M, int N, int K, bf16* out, int64_t ld_out,
             float* f32, int kind, int* status, uint64_t limit, cudaStream_t st) {
  GemmParams g = gemm_base(status, limit);
  g.M = M;
  g.N = N;
  g.K = K;
  g.m_tiles = (M + 127) / 128;
  g.n_tiles = N / 128;
  g.k_blocks = (K + 63) / 64;
  g.out = out;
  g.ld_out = ld_out;
  g.carry = f32;
  g.carry_in = 0;
  g.final_out = out != nullptr;
  UPIPE_LAUNCH(kind, launch_gemm(GK_OPROJ, ma, mb, g, st));
  return UPIPE_OK;
}

// C = A B, A [M, K] K-major, B [K, N] with N contiguous: bf16 out.
int gemm_ab(const CUtensorMap& ma, const CUtensorMap& mb_mn, int M, int N, int K, bf16* out, int64_t ld_out,
            int kind, int* status, uint64_t limit, cudaStream_t st) {
  GemmParams g = gemm_base(status, limit);
  g.M = M;
  g.N = N;
  g.K = K;
  g.m_tiles = (M + 127) / 128;
  g.n_tiles = N / 128;
  g.k_blocks = (K + 63) / 64;
  g.out = out;
  g.ld_out = ld_out;
  UPIPE_LAUNCH(kind, launch_gemm(GK_NN, ma, mb_mn, g, st));
  return UPIPE_OK;
}

// C (+)= A^T B over the K = `rows` tokens of one tile: A [rows, M] and
// B [rows, N] (M / N contiguous); fp32 C [M, N] carried in place.
int gemm_wgrad(const CUtensorMap& ma_mn, const CUtensorMap& mb_mn, int M, int N, int rows, float* C,
               bool carry_in, int* status, uint64_t limit, cudaStream_t st) {
  GemmParams g = gemm_base(status, limit);
  g.M = M;
  g.N = N;
  g.K = rows;
  g.m_tiles = M / 128;
  g.n_tiles = N / 128;
  g.k_blocks = (rows + 63) / 64;
  g.carry = C;
  g.carry_in = carry_in ? 1 : 0;
  g.final_out = 0;
  UPIPE_LAUNCH(UPIPE_KIND_ALST_WGRAD, launch_gemm(GK_WGRAD, ma_mn, mb_mn, g, st));
  return UPIPE_OK;
}

}  // namespace

cudaError_t launch_ce_rows(const float* z, int64_t ld_z, int V, const int32_t* labels, float scale, float* loss,
                           __nv_bfloat16* dz, int64_t ld_dz, int rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  ce_rows_kernel<<<rows, kCeThreads, 0, s>>>(z, ld_z, V, labels, scale, loss, dz, ld_dz);
  return cudaGetLastError();
}

}  // namespace upipe

using namespace upipe;

extern "C" {

size_t upipe_mlp_workspace_bytes(const upipe_mlp_cfg* cfg, int pass) {
  MlpShape s;
  if ((pass != 0 && pass != 1) || !check_mlp(cfg, &s)) return 0;
  return mlp_plan(s, pass).total;
}

int upipe_mlp_fwd(const upipe_mlp_cfg* cfg, const uint16_t* x, const uint16_t* Wgu, const uint16_t* Wd, uint16_t* y,
                  void* ws, size_t ws_bytes, void* stream) {
  MlpShape s;
  if (!check_mlp(cfg, &s) || !x || !Wgu || !Wd || !y || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wgu) || !aligned16(Wd) || !aligned16(y) || !aligned16(ws))
    return UPIPE_ERR_INVALID_ARG;
  const MlpPlan pl = mlp_plan(s, 0);
  if (ws_bytes < pl.total) return UPIPE_ERR_WS_TOO_SMALL;
  int* status = nullptr;
  if (int e = device_ready(&status)) return e;
  const uint64_t limit = spin_limit_ns();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bf16* H = reinterpret_cast<bf16*>(static_cast<uint8_t*>(ws) + pl.off_h);
  const int D = s.D, F = s.F;
  CUtensorMap m_wgu, m_wd, m_h;
  UPIPE_MAP(map2d(&m_wgu, Wgu, D, 2ull * F, D, 128));
  UPIPE_MAP(map2d(&m_wd, Wd, F, D, F, 128));
  for (int64_t r0 = 0; r0 < s.L; r0 += s.T) {
    const int rows = static_cast<int>(s.L - r0 < s.T ? s.L - r0 : s.T);
    CUtensorMap m_x;
    UPIPE_MAP(map2d(&m_x, x + r0 * D, D, rows, D, 128));
    UPIPE_MAP(map2d(&m_h, H, F, rows, F, 128));
    // H = silu(x Wg^T) * (x Wu^T)
    GemmParams g = gemm_base(status, limit);
    g.M = rows;
    g.N = 2 * F;
    g.K = D;
    g.m_tiles = (rows + 127) / 128;
    g.n_tiles = 2 * F / 128;
    g.k_blocks = D / 64;
    g.b_col0 = F;
    g.out = H;
    g.ld_out = F;
    UPIPE_LAUNCH(UPIPE_KIND_ALST_GU, launch_gemm(GK_GU, m_x, m_wgu, g, st));
    // y = H Wd^T
    if (int e = gemm_abt(m_h, m_wd, rows, D, F, reinterpret_cast<bf16*>(y) + r0 * D, D, nullptr,
                         UPIPE_KIND_ALST_GEMM, status, limit, st))
      return e;
  }
  return UPIPE_OK;
}

int upipe_mlp_bwd(const upipe_mlp_cfg* cfg, const uint16_t* x, const uint16_t* Wgu, const uint16_t* Wd,
                  const uint16_t* dy, uint16_t* dx, float* dWgu, float* dWd, void* ws, size_t ws_bytes,
                  void* stream) {
  MlpShape s;
  if (!check_mlp(cfg, &s) || !x || !Wgu || !Wd || !dy || !dx || !dWgu || !dWd || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wgu) || !aligned16(Wd) || !aligned16(dy) || !aligned16(dx) || !aligned16(dWgu) ||
      !aligned16(dWd) || !aligned16(ws))
    return UPIPE_ERR_INVALID_ARG;
  const MlpPlan pl = mlp_plan(s, 1);
  if (ws_bytes < pl.total) return UPIPE_ERR_WS_TOO_SMALL;
  int* status = nullptr;
  if (int e = device_ready(&status)) return e;
  const uint64_t limit = spin_limit_ns();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  bf16* H = reinterpret_cast<bf16*>(w + pl.off_h);
  bf16* dH = reinterpret_cast<bf16*>(w + pl.off_dh);
  bf16* dGU = reinterpret_cast<bf16*>(w + pl.off_dgu);
  const int D = s.D, F = s.F;
  CUtensorMap m_wgu, m_wgu_mn, m_wd_mn;
  UPIPE_MAP(map2d(&m_wgu, Wgu, D, 2ull * F, D, 128));
  UPIPE_MAP(map2d(&m_wgu_mn, Wgu, D, 2ull * F, D, 64));  // B of dx = dGU Wgu: [K = 2F, N = D]
  UPIPE_MAP(map2d(&m_wd_mn, Wd, F, D, F, 64));           // B of dH = dy Wd: [K = D, N = F]
  int tile = 0;
  for (int64_t r0 = 0; r0 < s.L; r0 += s.T, ++tile) {
    const int rows = static_cast<int>(s.L - r0 < s.T ? s.L - r0 : s.T);
    CUtensorMap m_x, m_x_mn, m_dy, m_dy_mn, m_h_mn, m_dgu, m_dgu_mn;
    UPIPE_MAP(map2d(&m_x, x + r0 * D, D, rows, D, 128));
    UPIPE_MAP(map2d(&m_x_mn, x + r0 * D, D, rows, D, 64));
    UPIPE_MAP(map2d(&m_dy, dy + r0 * D, D, rows, D, 128));
    UPIPE_MAP(map2d(&m_dy_mn, dy + r0 * D, D, rows, D, 64));
    UPIPE_MAP(map2d(&m_h_mn, H, F, rows, F, 64));
    UPIPE_MAP(map2d(&m_dgu, dGU, 2ull * F, rows, 2ull * F, 128));
    UPIPE_MAP(map2d(&m_dgu_mn, dGU, 2ull * F, rows, 2ull * F, 64));
    // dH = dy Wd
    if (int e = gemm_ab(m_dy, m_wd_mn, rows, F, D, dH, F, UPIPE_KIND_ALST_GEMM, status, limit, st)) return e;
    // recompute g, u: H and [dG | dU] from dH
    GemmParams g = gemm_base(status, limit);
    g.M = rows;
    g.N = 2 * F;
    g.K = D;
    g.m_tiles = (rows + 127) / 128;
    g.n_tiles = 2 * F / 128;
    g.k_blocks = D / 64;
    g.b_col0 = F;
    g.out = H;
    g.ld_out = F;
    g.in2 = dH;
    g.ld_in2 = F;
    g.out2 = dGU;
    g.ld_out2 = 2 * F;
    UPIPE_LAUNCH(UPIPE_KIND_ALST_GU, launch_gemm(GK_GU_BWD, m_x, m_wgu, g, st));
    // dWd (+)= dy^T H, dWgu (+)= [dG | dU]^T x
    if (int e = gemm_wgrad(m_dy_mn, m_h_mn, D, F, rows, dWd, tile > 0, status, limit, st)) return e;
    if (int e = gemm_wgrad(m_dgu_mn, m_x_mn, 2 * F, D, rows, dWgu, tile > 0, status, limit, st)) return e;
    // dx = [dG | dU] Wgu
    if (int e = gemm_ab(m_dgu, m_wgu_mn, rows, D, 2 * F, reinterpret_cast<bf16*>(dx) + r0 * D, D,
                        UPIPE_KIND_ALST_GEMM, status, limit, st))
      return e;
  }
  return UPIPE_OK;
}

int upipe_mlp_choose_t(const upipe_mlp_cfg* cfg, size_t budget_bytes, int pass) {
  MlpShape s;
  if ((pass < 0 || pass > 2) || !cfg) return UPIPE_ERR_INVALID_ARG;
  upipe_mlp_cfg c = *cfg;
  c.T = 128;
  if (!check_mlp(&c, &s)) return UPIPE_ERR_INVALID_ARG;
  // Bytes grow linearly with T; a tile never needs to exceed L rows.
  const int64_t t_max = (s.L + 127) / 128 * 128;
  const size_t per128 = mlp_plan(s, pass == 0 ? 0 : 1).total;  // T = 128: aligned to 1 KiB per buffer
  if (per128 > budget_bytes) return UPIPE_ERR_WS_TOO_SMALL;
  int64_t best = 128;
  for (int64_t t = 128; t <= t_max && t <= 0x7fffff80LL; t += 128) {
    s.T = static_cast<int>(t);
    if (mlp_plan(s, pass == 0 ? 0 : 1).total > budget_bytes) break;
    best = t;
  }
  return static_cast<int>(best);
}

int upipe_ce_choose_t(const upipe_ce_cfg* cfg, size_t budget_bytes) {
  CeShape s;
  if (!cfg) return UPIPE_ERR_INVALID_ARG;
  upipe_ce_cfg c = *cfg;
  c.T = 128;
  if (!check_ce(&c, &s)) return UPIPE_ERR_INVALID_ARG;
  if (ce_total(s) > budget_bytes) return UPIPE_ERR_WS_TOO_SMALL;
  const int64_t t_max = (s.L + 127) / 128 * 128;
  int64_t best = 128;
  for (int64_t t = 128; t <= t_max && t <= 0x7fffff80LL; t += 128) {
    s.T = static_cast<int>(t);
    if (ce_total(s) > budget_bytes) break;
    best = t;
  }
  return static_cast<int>(best);
}

size_t upipe_ce_workspace_bytes(const upipe_ce_cfg* cfg) {
  CeShape s;
  if (!check_ce(cfg, &s)) return 0;
  return ce_total(s);
}

int upipe_ce_fwd_bwd(const upipe_ce_cfg* cfg, const uint16_t* h, const uint16_t* W, const int32_t* labels,
                     float scale, float* loss, uint16_t* dh, float* dW, void* ws, size_t ws_bytes, void* stream) {
  CeShape s;
  if (!check_ce(cfg, &s) || !h || !W || !labels || !loss || !dh || !dW || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(W) || !aligned16(labels) || !aligned16(loss) || !aligned16(dh) || !aligned16(dW) ||
      !aligned16(ws) || !std::isfinite(scale))
    return UPIPE_ERR_INVALID_ARG;
  if (ws_bytes < ce_total(s)) return UPIPE_ERR_WS_TOO_SMALL;
  int* status = nullptr;
  if (int e = device_ready(&status)) return e;
  const uint64_t limit = spin_limit_ns();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* Z = static_cast<float*>(ws);
  bf16* dZ = reinterpret_cast<bf16*>(static_cast<uint8_t*>(ws) + ce_z_bytes(s));
  const int D = s.D, V = s.V;
  CUtensorMap m_w, m_w_mn;
  UPIPE_MAP(map2d(&m_w, W, D, V, D, 128));
  UPIPE_MAP(map2d(&m_w_mn, W, D, V, D, 64));  // B of dh = dZ W: [K = V, N = D]
  int tile = 0;
  for (int64_t r0 = 0; r0 < s.L; r0 += s.T, ++tile) {
    const int rows = static_cast<int>(s.L - r0 < s.T ? s.L - r0 : s.T);
    CUtensorMap m_h, m_h_mn, m_dz, m_dz_mn;
    UPIPE_MAP(map2d(&m_h, h + r0 * D, D, rows, D, 128));
    UPIPE_MAP(map2d(&m_h_mn, h + r0 * D, D, rows, D, 64));
    UPIPE_MAP(map2d(&m_dz, dZ, V, rows, V, 128));
    UPIPE_MAP(map2d(&m_dz_mn, dZ, V, rows, V, 64));
    // Z = h W^T (fp32)
    if (int e = gemm_abt(m_h, m_w, rows, V, D, nullptr, 0, Z, UPIPE_KIND_ALST_GEMM, status, limit, st)) return e;
    // per-row LSE, loss, dZ
    UPIPE_LAUNCH(UPIPE_KIND_CE_ROWS, launch_ce_rows(Z, V, V, labels + r0, scale, loss + r0, dZ, V, rows, st));
    // dh = dZ W, dW (+)= dZ^T h
    if (int e = gemm_ab(m_dz, m_w_mn, rows, D, V, reinterpret_cast<bf16*>(dh) + r0 * D, D, UPIPE_KIND_ALST_GEMM,
                        status, limit, st))
      return e;
    if (int e = gemm_wgrad(m_dz_mn, m_h_mn, V, D, rows, dW, tile > 0, status, limit, st)) return e;
  }
  return UPIPE_OK;
}

}  // extern "C"
