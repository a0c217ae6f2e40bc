// Parameter blocks shared by the host orchestration (upipe.cu) and the
// kernels (gemm.cu, attn_fwd.cu, attn_bwd.cu, aux.cu).  Plain structs of
// scalars and pointers, passed by value as __grid_constant__ kernel params.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

// Device status bits (the library's status word).
#define UPIPE_STATUS_TIMEOUT 1        // a bounded wait ran out
#define UPIPE_STATUS_DRAIN_TIMEOUT 2  // unwinding after a timeout also ran out

namespace upipe {

constexpr int kHeadDim = 128;     // d: one head = one 128-wide MMA tile
constexpr int kMaxSlots = 96;     // H + 2 Hkv limit (per-slot tables below)

// ------------------------------------------------------------------ GEMMs
//
// One tcgen05 GEMM kernel (persistent CTA pairs, 256x256 output tiles, K
// blocks of 64) serves the six projection contractions of the layer and the
// contractions of the sequence-tiled MLP and loss.  The kind fixes which
// operands are K-major or MN-major, how tile coordinates map to tensor
// coordinates and what the epilogue does.
enum GemmKind : int {
  GK_QKV = 0,    // Y_c = x W_c^T, fused RoPE + bf16 cast into head-major Q/K/V
  GK_OPROJ = 1,  // out32 (+)= O_c Wo[:, cols_c]^T with an fp32 carry
  GK_DO = 2,     // dO_c = dout Wo[:, cols_c]; also Delta = rowsum(dO * O)
  GK_DWO = 3,    // dWo[:, cols_c] = dout^T O_c (fp32)
  GK_DWQKV = 4,  // dWqkv[rows_c] = dqkv_c^T x (fp32)
  GK_DX = 5,     // dx32 (+)= dqkv_c W_c with an fp32 carry
  // Sequence-tiled MLP and loss.  GK_OPROJ also serves them as a plain
  // A B^T (both K-major): bf16 out (final_out) or fp32 out (no carry_in).
  GK_GU = 6,      // H = silu(X Wg^T) * (X Wu^T) -> bf16 [M, F]; B = Wgu [2F, K], b_col0 = F
  GK_GU_BWD = 7,  // from X Wgu^T and dH (in2): H -> out, [dG | dU] -> out2 (bf16 [M, 2F])
  GK_NN = 8,      // C = A B, A [M, K] K-major, B [K, N] (N contiguous) -> bf16 [M, N]
  GK_WGRAD = 9,   // C (+)= A^T B, A [K, M], B [K, N] (both M/N contiguous), fp32 C in `carry` [M, N]
};

struct GemmParams {
  int M, N, K;
  int m_tiles, n_tiles, k_blocks;
  int a_col0, b_col0;          // element offsets added to the column coordinate
  int out_col0;                // DWO: first output column
  int L;                       // rows of head-major buffers
  int16_t tab0[kMaxSlots];     // QKV: n tile -> W row block; DWQKV: m tile -> A slot; DX: K slot -> A slot
  int16_t tab1[kMaxSlots];     // DWQKV: m tile -> dWqkv row block; DX: K slot -> W row block
  void* out;                   // see GemmKind
  int64_t ld_out;              // elements
  float* carry;                // OPROJ / DX: fp32 [M, N]
  int carry_in;                // accumulator starts from the carry
  int final_out;               // write bf16 `out` (else write the fp32 carry)
  int rope_slots;              // QKV: slots below this are rotated
  const float2* rope;          // [L, 64] (cos, sin)
  const __nv_bfloat16* o_rows; // DO: O_c rows for Delta
  int64_t ld_o;
  const float* lse_in;         // DO: the chunk's LSE rows [U, L]
  float* ld_rec;               // DO: per 64-query tile records (see AttnBwdParams::ld)
  int lo_z;                    // DWQKV / DX: A slot offset of the low bf16 halves (0 = no split)
  int k_mid;                   // DWQKV: > 0 splits K into blocks [0, k_mid) and [k_mid, k_blocks), two
                               // work units per tile that add into the zeroed output (fp32 reductions)
  const __nv_bfloat16* in2;    // GU_BWD: dH [M, F]
  int64_t ld_in2;
  __nv_bfloat16* out2;         // GU_BWD: [dG | dU] [M, 2F]
  int64_t ld_out2;
  int* status;
  uint64_t limit_ns;
};

// -------------------------------------------------------------- attention
//
// Q, K, V (and dO) are read through 3-D tensor maps {d, L, heads}; the z
// coordinate of local head h is q_z0 + h, of its KV head k_z0 + h / g_loc.
// Forward attention modes (see attn_fwd.cu).
enum AttnFwdMode : int {
  kOnline = 0,   // online softmax: O and LSE
  kLseIn = 1,    // LSE given (lse_in): O from the final probabilities
  kLseOnly = 2,  // LSE only
};

struct AttnFwdParams {
  int mode;     // AttnFwdMode
  int L;
  int nheads;   // query heads in this launch
  int g_loc;    // query heads per KV head in this launch
  int q_z0, k_z0, v_z0;
  __nv_bfloat16* o;  // O of local head h, row p: o + p*o_row + h*o_head
  int64_t o_row, o_head;
  float* lse;        // [nheads, L]; kOnline (when write_lse) and kLseOnly write it
  int write_lse;
  const float* lse_in;  // kLseIn: [nheads, L], natural log
  float scale_log2;  // log2(e) / sqrt(d)
  int* status;
  uint64_t limit_ns;
};

struct AttnBwdParams {
  int L;
  int nheads;   // query heads in this launch
  int g_loc;    // query heads per KV head in this launch
  int nkv;      // KV heads in this launch
  int q_z0, k_z0, v_z0, do_z0;
  // Per local head h and 64-query tile t, a 128-float record at
  // ld + (h * ceil(L/64) + t) * 128: -LSE * log2(e) of the tile's 64 queries
  // (-inf past L), then their Delta = rowsum(dO * O) (0 past L).
  const float* ld;
  float scale;         // 1/sqrt(d)
  float scale_log2;    // log2(e)/sqrt(d)
  __nv_bfloat16* dq;   // dQ of local head h, row p: dq + p*dq_row + h*dq_head
  int64_t dq_row, dq_head;
  __nv_bfloat16* dk;   // dK/dV of local KV head j, row p: d? + p*dkv_row + j*dkv_head
  __nv_bfloat16* dv;
  int64_t dkv_row, dkv_head;
  int64_t lo_off;      // > 0: also write x - bf16(x) as bf16 at (pointer + lo_off)
  float* dkv_carry;    // [nkv][2][L][d] fp32: the dK then dV partial sums
  int carry_in;        // start dK/dV from the carry
  int carry_out;       // write the carry instead of the bf16 dK/dV
  const float2* rope;  // rotate dQ and dK back by -angle when non-null
  int* status;
  uint64_t limit_ns;
};

// While an object of this type lives, launches made by the current host
// thread record no profiling events (the entry point that allocates nothing
// must not create events or grow host vectors).
class ProfilingOff {
 public:
  ProfilingOff();
  ~ProfilingOff();
  ProfilingOff(const ProfilingOff&) = delete;
  ProfilingOff& operator=(const ProfilingOff&) = delete;

 private:
  bool prev_;
};

// ------------------------------------------------------------- launchers

cudaError_t launch_gemm(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                        cudaStream_t s);
cudaError_t launch_attn_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const AttnFwdParams& p, int n_qblocks, cudaStream_t s);
// All maps of the two backward kernels have 128-row boxes.
cudaError_t launch_attn_bwd_dq(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& dO, const AttnBwdParams& p, int n_qblocks, cudaStream_t s);
cudaError_t launch_attn_bwd_dkdv(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& dO, const AttnBwdParams& p, int n_kblocks, cudaStream_t s);
cudaError_t launch_rope_table(float2* table, int64_t L, double theta, cudaStream_t s);
// Writes the LSE/Delta records of AttnBwdParams::ld for `nheads` heads.
cudaError_t launch_delta(const __nv_bfloat16* o, int64_t o_row, int64_t o_head, const __nv_bfloat16* dO,
                         int64_t do_row, int64_t do_head, const float* lse, float* ld, int64_t L, int nheads,
                         cudaStream_t s);
// Zeroes the fp32 rows [128 b, 128 b + 128) x [0, cols) of `base` (leading
// dimension ld) for the n row blocks b listed in `blocks`.
cudaError_t launch_zero_rows(float* base, int64_t ld, int cols, const int16_t* blocks, int n, cudaStream_t s);
cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t s);
// Cross-entropy rows: for each of the `rows` rows of the fp32 logits z
// (leading dimension ld_z, V columns), LSE, the row's loss (0 for a negative
// label) and dz = scale (softmax - onehot) as bf16 (leading dimension ld_dz;
// a row of zeros for a negative label).
cudaError_t launch_ce_rows(const float* z, int64_t ld_z, int V, const int32_t* labels, float scale, float* loss,
                           __nv_bfloat16* dz, int64_t ld_dz, int rows, cudaStream_t s);

}  // namespace upipe
