// C ABI of the head-chunked attention layer: argument checks, the chunk
// planner / workspace carve-up, TMA tensor maps and the per-chunk launch
// sequence.  Everything here runs on the host and only enqueues kernels on
// the caller's stream.
//
// The chunk loop follows "Untied Ulysses Pushes Llama-3-8B Training to 5
// Million Tokens" (talk write-up), paragraph on intermediate buffers: one
// group of heads is projected and run through attention, its partial result
// is added into the output, and the next group reuses the same buffers.  The
// workspace offsets below are computed once per call and are identical for
// every chunk.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <initializer_list>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "host.h"
#include "upipe.h"
#include "upipe_internal.h"

// Device status word of this library (one per device that loads it).
__device__ int g_upipe_status;

namespace upipe {
namespace {

constexpr size_t kAlign = 1024;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Shape {
  int64_t L;
  int D, H, Hkv, d, U, g, kvc, nch;
};

// Validates cfg; `layer` adds the projection constraints.
bool check_cfg(const upipe_cfg* c, bool layer, Shape* s) {
  if (!c) return false;
  if (c->L < 1 || c->L > 0x7fffffffLL) return false;
  if (c->d != kHeadDim || c->causal != 1) return false;
  if (c->H < 1 || c->Hkv < 1 || c->H % c->Hkv != 0) return false;
  if (c->H + 2 * c->Hkv > kMaxSlots) return false;
  if (c->U < 1 || c->H % c->U != 0) return false;
  const int g = c->H / c->Hkv;
  if (c->U % g != 0 && g % c->U != 0) return false;
  if (layer) {
    if (c->D < 128 || c->D % 128 != 0) return false;
    if (!(c->rope_theta > 0.0) || !std::isfinite(c->rope_theta)) return false;
  }
  s->L = c->L;
  s->D = c->D;
  s->H = c->H;
  s->Hkv = c->Hkv;
  s->d = c->d;
  s->U = c->U;
  s->g = g;
  s->kvc = c->U >= g ? c->U / g : 1;
  s->nch = c->H / c->U;
  return true;
}

// Workspace carve-up.  Offsets are relative to ws; a zero size means absent.
struct Plan {
  size_t rope = 0, qkv = 0, o = 0, dO = 0, delta = 0, dqkv = 0, dkv_carry = 0, carry32 = 0;
  size_t off_rope = 0, off_qkv = 0, off_o = 0, off_dO = 0, off_delta = 0, off_dqkv = 0, off_dkv = 0, off_carry = 0;
  size_t total = 0;
  size_t chunk_bytes() const { return qkv + o + dO + delta + dqkv + dkv_carry; }
  size_t fixed_bytes() const { return carry32 + rope; }
};

// Where the layer entries keep the attention output O between the forward
// and the backward.
enum OMode {
  kOWorkspace = 0,  // O_c lives in the workspace; the backward recomputes it
  kODevice = 1,     // the caller's o_saved [L, H*128] holds every chunk's O
  kOHost = 2,       // page-locked host memory holds it; chunk buffers stage the copies
                    // (three in the forward, two in the backward)
};

// LSE/Delta records of the backward: per head of the chunk and 64-query
// tile, 64 -LSE*log2(e) then 64 Delta floats.
size_t ld_records_bytes(const Shape& s) {
  return static_cast<size_t>(s.U) * static_cast<size_t>((s.L + 63) / 64) * 128 * sizeof(float);
}

Plan make_plan(const Shape& s, int pass, bool core, int o_mode) {
  Plan p;
  const size_t L = static_cast<size_t>(s.L);
  const size_t slot = L * kHeadDim * 2;  // one head-major [L, 128] bf16 buffer
  const bool carry_kv = s.U < s.g;       // dK/dV carried across the chunks of a group
  if (core) {
    if (pass == 1) {
      p.delta = ld_records_bytes(s);
      if (carry_kv) p.dkv_carry = 2 * L * kHeadDim * 4;
    }
  } else {
    p.rope = L * 64 * sizeof(float2);
    p.qkv = (s.U + 2 * s.kvc) * slot;
    if (o_mode == kOWorkspace) p.o = s.U * slot;
    if (o_mode == kOHost) p.o = (pass == 0 ? 3 : 2) * s.U * slot;
    if (s.nch > 1) p.carry32 = L * s.D * 4;
    if (pass == 1) {
      p.dO = s.U * slot;
      p.delta = ld_records_bytes(s);
      p.dqkv = 2 * (s.U + 2 * s.kvc) * slot;  // high then low bf16 halves
      if (carry_kv) p.dkv_carry = 2 * L * kHeadDim * 4;
    }
  }
  size_t off = 0;
  auto take = [&](size_t bytes, size_t* o) {
    *o = off;
    off += align_up(bytes);
  };
  take(p.rope, &p.off_rope);
  take(p.qkv, &p.off_qkv);
  take(p.o, &p.off_o);
  take(p.dO, &p.off_dO);
  take(p.delta, &p.off_delta);
  take(p.dqkv, &p.off_dqkv);
  take(p.dkv_carry, &p.off_dkv);
  take(p.carry32, &p.off_carry);
  p.total = off;
  return p;
}

}  // namespace

// ------------------------------------------- helpers shared through host.h

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

uint64_t spin_limit_ns() {
  const char* e = std::getenv("UPIPE_SPIN_LIMIT_NS");
  if (e && *e) {
    char* end = nullptr;
    unsigned long long v = std::strtoull(e, &end, 10);
    if (end && *end == 0) return v;
  }
  return 2000000000ull;
}

// Device checks and the status word address, cached per device.  The first
// call on a device fills its entry under a lock; later calls read it through
// an acquire load, so calls from several host threads see a complete entry.
constexpr int kMaxDev = 64;
std::atomic<int> g_dev_state[kMaxDev];  // 0 unknown, 1 ok, -1 unsupported
int* g_status_ptr[kMaxDev];
std::mutex g_dev_mu;

int device_ready(int** status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UPIPE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDev) return UPIPE_ERR_UNSUPPORTED_DEVICE;
  if (g_dev_state[dev].load(std::memory_order_acquire) == 0) {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (g_dev_state[dev].load(std::memory_order_relaxed) == 0) {
      int major = 0, minor = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return UPIPE_ERR_CUDA;
      if (major != 10 || minor != 3) {
        g_dev_state[dev].store(-1, std::memory_order_release);
      } else {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_upipe_status) != cudaSuccess) return UPIPE_ERR_CUDA;
        g_status_ptr[dev] = static_cast<int*>(ptr);
        g_dev_state[dev].store(1, std::memory_order_release);
      }
    }
  }
  if (g_dev_state[dev].load(std::memory_order_acquire) < 0) return UPIPE_ERR_UNSUPPORTED_DEVICE;
  *status = g_status_ptr[dev];
  return UPIPE_OK;
}

// ------------------------------------------------------------ tensor maps

// Looked up once (a function-local static is initialised exactly once, even
// when several threads arrive together).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// bf16 [rows, cols] with leading dimension ld (elements); box 64 x box_rows.
bool map2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 heads of 128: element (c, row, head) at base + row*row_stride + head*head_stride.
bool map3d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t heads, uint64_t row_stride,
           uint64_t head_stride, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {kHeadDim, rows, heads};
  cuuint64_t strides[2] = {row_stride * 2, head_stride * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch accounting: a counter of every kernel launch, and optional CUDA
// event pairs recorded around each launch on the launching stream.  A host
// thread inside the entry point that allocates nothing records no events
// (an event pair may need cudaEventCreate and grows a host vector).
std::atomic<int64_t> g_launches{0};
std::atomic<bool> g_profile{false};
thread_local bool t_no_profile = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pool_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// See upipe_internal.h.
ProfilingOff::ProfilingOff() : prev_(t_no_profile) { t_no_profile = true; }
ProfilingOff::~ProfilingOff() { t_no_profile = prev_; }

namespace {

// dQ and dK/dV of one chunk run concurrently: neither reads what the other
// writes.  dK/dV goes to a second stream of the device's greatest priority,
// so its CTAs (few, long: key tile kb sees L - 128 kb queries of g_loc
// heads) are dispatched first, and dQ's many short CTAs, heaviest first,
// fill the SMs that the dK/dV tail leaves idle.  The stream and its fork /
// join events are created on the first call per device.
struct Side {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
Side g_side[kMaxDev];
// Serialises the fork / launch / join sequence: the fork and join events are
// shared, and a stream wait takes the event as last recorded, so two host
// threads interleaving their sequences could join the wrong work.
std::mutex g_side_mu;

int side_stream(Side** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UPIPE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDev) return UPIPE_ERR_UNSUPPORTED_DEVICE;
  Side& sd = g_side[dev];
  if (!sd.join) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return UPIPE_ERR_CUDA;
    if (!sd.s && cudaStreamCreateWithPriority(&sd.s, cudaStreamNonBlocking, greatest) != cudaSuccess)
      return UPIPE_ERR_CUDA;
    if (!sd.fork && cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess) return UPIPE_ERR_CUDA;
    if (cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess) return UPIPE_ERR_CUDA;
  }
  *out = &sd;
  return UPIPE_OK;
}

int launch_attn_bwd_pair(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mdo, const AttnBwdParams& b, int m_tiles, cudaStream_t st) {
  std::lock_guard<std::mutex> lock(g_side_mu);
  Side* sd = nullptr;
  if (int e = side_stream(&sd)) return e;
  UPIPE_CU(cudaEventRecord(sd->fork, st));
  UPIPE_CU(cudaStreamWaitEvent(sd->s, sd->fork, 0));
  UPIPE_CU(counted(UPIPE_KIND_ATTN_BWD_DKDV, sd->s, [&] { return launch_attn_bwd_dkdv(mq, mk, mv, mdo, b, m_tiles, sd->s); }));
  UPIPE_CU(counted(UPIPE_KIND_ATTN_BWD_DQ, st, [&] { return launch_attn_bwd_dq(mq, mk, mv, mdo, b, m_tiles, st); }));
  UPIPE_CU(cudaEventRecord(sd->join, sd->s));
  UPIPE_CU(cudaStreamWaitEvent(st, sd->join, 0));
  return UPIPE_OK;
}

// Copy streams of the activation offload: one per direction and device,
// created on first use, with an event to order each batch of copies after
// the caller's stream and one per direction to join them back.  o_ready and
// o_done[3] order the layer entries' copies of O to and from host memory
// (o_done[b]: the last copy through chunk buffer b).
struct Copier {
  cudaStream_t d2h = nullptr, h2d = nullptr;
  cudaEvent_t after = nullptr, done_d2h = nullptr, done_h2d = nullptr;
  cudaEvent_t o_ready = nullptr, o_done[3] = {nullptr, nullptr, nullptr};
};
Copier g_copier[kMaxDev];
std::mutex g_copier_mu;

int copier(Copier** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UPIPE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDev) return UPIPE_ERR_UNSUPPORTED_DEVICE;
  Copier& c = g_copier[dev];
  if (!c.done_h2d) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return UPIPE_ERR_CUDA;
    if (!c.d2h && cudaStreamCreateWithPriority(&c.d2h, cudaStreamNonBlocking, least) != cudaSuccess)
      return UPIPE_ERR_CUDA;
    if (!c.h2d && cudaStreamCreateWithPriority(&c.h2d, cudaStreamNonBlocking, least) != cudaSuccess)
      return UPIPE_ERR_CUDA;
    if (!c.after && cudaEventCreateWithFlags(&c.after, cudaEventDisableTiming) != cudaSuccess) return UPIPE_ERR_CUDA;
    for (cudaEvent_t* e : {&c.done_d2h, &c.o_ready, &c.o_done[0], &c.o_done[1], &c.o_done[2]})
      if (!*e && cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return UPIPE_ERR_CUDA;
    if (cudaEventCreateWithFlags(&c.done_h2d, cudaEventDisableTiming) != cudaSuccess) return UPIPE_ERR_CUDA;
  }
  *out = &c;
  return UPIPE_OK;
}

// One copy on the direction's copy stream, after the caller's stream.
int async_copy(void* dst, const void* src, size_t bytes, bool to_host, cudaStream_t st) {
  if (bytes == 0) return UPIPE_OK;
  if (!dst || !src) return UPIPE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_copier_mu);
  Copier* c = nullptr;
  if (int e = copier(&c)) return e;
  cudaStream_t cs = to_host ? c->d2h : c->h2d;
  if (cudaEventRecord(c->after, st) != cudaSuccess || cudaStreamWaitEvent(cs, c->after, 0) != cudaSuccess)
    return UPIPE_ERR_CUDA;
  if (cudaMemcpyAsync(dst, src, bytes, to_host ? cudaMemcpyDeviceToHost : cudaMemcpyHostToDevice, cs) !=
      cudaSuccess)
    return UPIPE_ERR_CUDA;
  return UPIPE_OK;
}


// Page-locked (or registered) host memory: the only kind a copy stream
// copies without blocking the calling thread.
bool host_pinned(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

// One chunk's O ([L, U*128] bf16) between a workspace buffer and its block
// of host memory, on the direction's copy stream after everything enqueued
// on st so far; o_done[buf] marks its end.
int copy_o_chunk(Copier* cp, void* dst, const void* src, size_t bytes, bool to_host, int buf, cudaStream_t st) {
  cudaStream_t cs = to_host ? cp->d2h : cp->h2d;
  if (cudaEventRecord(cp->o_ready, st) != cudaSuccess || cudaStreamWaitEvent(cs, cp->o_ready, 0) != cudaSuccess ||
      cudaMemcpyAsync(dst, src, bytes, to_host ? cudaMemcpyDeviceToHost : cudaMemcpyHostToDevice, cs) !=
          cudaSuccess ||
      cudaEventRecord(cp->o_done[buf], cs) != cudaSuccess)
    return UPIPE_ERR_CUDA;
  return UPIPE_OK;
}

using bf16 = __nv_bfloat16;

// Chunk c: query heads [c*U, (c+1)*U); first KV head and W row blocks.
struct Chunk {
  int q0, kv0;
};
Chunk chunk_of(const Shape& s, int c) { return Chunk{c * s.U, (c * s.U) / s.g}; }

// W row block (units of 128 rows) of slot `sl` of chunk c: q slots, k, v.
int w_block(const Shape& s, const Chunk& ch, int sl) {
  if (sl < s.U) return ch.q0 + sl;
  if (sl < s.U + s.kvc) return s.H + ch.kv0 + (sl - s.U);
  return s.H + s.Hkv + ch.kv0 + (sl - s.U - s.kvc);
}

// Layer forward; at most one of o_saved (device) and o_host (page-locked
// host memory) is non-null.
int layer_fwd(const upipe_cfg* cfg, const uint16_t* x, const uint16_t* Wqkv, const uint16_t* Wo, uint16_t* out,
              float* lse, uint16_t* o_saved, uint16_t* o_host, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  if (!check_cfg(cfg, true, &s)) return UPIPE_ERR_INVALID_ARG;
  if (!x || !Wqkv || !Wo || !out || !lse || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(out) || !aligned16(lse) ||
      !aligned16(ws) || (o_saved && !aligned16(o_saved)))
    return UPIPE_ERR_INVALID_ARG;
  const int o_mode = o_host ? kOHost : o_saved ? kODevice : kOWorkspace;
  const Plan pl = make_plan(s, 0, false, o_mode);
  if (ws_bytes < pl.total) return UPIPE_ERR_WS_TOO_SMALL;
  int* status = nullptr;
  if (int e = device_ready(&status)) return e;
  // The O copies use the shared copy streams and events: one call at a time.
  std::unique_lock<std::mutex> copy_lock;
  Copier* cp = nullptr;
  if (o_host) {
    copy_lock = std::unique_lock<std::mutex>(g_copier_mu);
    if (int e = copier(&cp)) return e;
  }
  const uint64_t limit = spin_limit_ns();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float2* rope = reinterpret_cast<float2*>(w + pl.off_rope);
  bf16* qkv = reinterpret_cast<bf16*>(w + pl.off_qkv);
  float* carry = reinterpret_cast<float*>(w + pl.off_carry);
  const int64_t L = s.L;
  const int slots = s.U + 2 * s.kvc;
  const int m_tiles = static_cast<int>((L + 127) / 128);

  UPIPE_LAUNCH(UPIPE_KIND_ROPE_TABLE, launch_rope_table(rope, L, cfg->rope_theta, st));

  CUtensorMap m_x, m_wqkv, m_qkv, m_o, m_wo;
  UPIPE_MAP(map2d(&m_x, x, s.D, L, s.D, 128));
  UPIPE_MAP(map2d(&m_wqkv, Wqkv, s.D, static_cast<uint64_t>(s.H + 2 * s.Hkv) * 128, s.D, 128));
  UPIPE_MAP(map3d(&m_qkv, qkv, L, slots, 128, L * 128, 128));
  const bf16* obuf = o_saved ? reinterpret_cast<const bf16*>(o_saved) : reinterpret_cast<bf16*>(w + pl.off_o);
  const int64_t ld_o = o_saved ? static_cast<int64_t>(s.H) * 128 : static_cast<int64_t>(s.U) * 128;
  const size_t o_chunk_elems = static_cast<size_t>(L) * s.U * 128;  // one chunk buffer of O
  UPIPE_MAP(map2d(&m_o, obuf, ld_o, L, ld_o, 128));
  // Host mode: three chunk buffers, so a chunk's copy to host has two
  // chunks' compute to finish before its buffer is reused.
  CUtensorMap m_ob[3];
  m_ob[0] = m_o;
  if (o_host) {
    UPIPE_MAP(map2d(&m_ob[1], obuf + o_chunk_elems, ld_o, L, ld_o, 128));
    UPIPE_MAP(map2d(&m_ob[2], obuf + 2 * o_chunk_elems, ld_o, L, ld_o, 128));
  }
  UPIPE_MAP(map2d(&m_wo, Wo, static_cast<uint64_t>(s.H) * 128, s.D, static_cast<uint64_t>(s.H) * 128, 128));

  for (int c = 0; c < s.nch; ++c) {
    const Chunk ch = chunk_of(s, c);
    // a-1/a-2: Q/K/V slice with fused RoPE.
    GemmParams g = gemm_base(status, limit);
    g.M = static_cast<int>(L);
    g.N = slots * 128;
    g.K = s.D;
    g.m_tiles = m_tiles;
    g.n_tiles = slots;
    g.k_blocks = s.D / 64;
    g.L = static_cast<int>(L);
    for (int sl = 0; sl < slots; ++sl) g.tab0[sl] = static_cast<int16_t>(w_block(s, ch, sl));
    g.out = qkv;
    g.rope_slots = s.U + s.kvc;
    g.rope = rope;
    UPIPE_LAUNCH(UPIPE_KIND_QKV_GEMM, launch_gemm(GK_QKV, m_x, m_wqkv, g, st));

    // a-3: causal attention.  A kept O is written from the final
    // probabilities (LSE first, then O from it): the same bits the
    // backward's recomputation of O produces.  O bound for host memory is
    // the online softmax's own output, staged in chunk buffer c % 3 once
    // the copy of chunk c - 3 has left it.
    const int buf = o_host ? c % 3 : 0;
    if (o_host && c >= 3) UPIPE_CU(cudaStreamWaitEvent(st, cp->o_done[buf], 0));
    AttnFwdParams a;
    std::memset(&a, 0, sizeof(a));
    a.L = static_cast<int>(L);
    a.nheads = s.U;
    a.g_loc = s.U / s.kvc;
    a.q_z0 = 0;
    a.k_z0 = s.U;
    a.v_z0 = s.U + s.kvc;
    a.o = const_cast<bf16*>(obuf) + (o_saved ? static_cast<int64_t>(ch.q0) * 128 : buf * o_chunk_elems);
    a.o_row = ld_o;
    a.o_head = 128;
    a.lse = lse + static_cast<int64_t>(ch.q0) * L;
    a.write_lse = 1;
    a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(128.0));
    a.status = status;
    a.limit_ns = limit;
    if (o_saved) {
      a.mode = kLseOnly;
      UPIPE_LAUNCH(UPIPE_KIND_ATTN_FWD, launch_attn_fwd(m_qkv, m_qkv, m_qkv, a, m_tiles, st));
      a.mode = kLseIn;
      a.lse_in = a.lse;
      a.write_lse = 0;
    }
    UPIPE_LAUNCH(UPIPE_KIND_ATTN_FWD, launch_attn_fwd(m_qkv, m_qkv, m_qkv, a, m_tiles, st));
    if (o_host) {
      if (int e = copy_o_chunk(cp, o_host + c * o_chunk_elems, a.o, o_chunk_elems * 2, true, buf, st)) return e;
    }

    // a-4: out32 (+)= O_c Wo[:, cols_c]^T; the last chunk writes bf16 out.
    GemmParams o = gemm_base(status, limit);
    o.M = static_cast<int>(L);
    o.N = s.D;
    o.K = s.U * 128;
    o.m_tiles = m_tiles;
    o.n_tiles = s.D / 128;
    o.k_blocks = s.U * 2;
    o.a_col0 = o_saved ? ch.q0 * 128 : 0;
    o.b_col0 = ch.q0 * 128;
    o.out = out;
    o.ld_out = s.D;
    o.carry = carry;
    o.carry_in = c > 0;
    o.final_out = c == s.nch - 1;
    UPIPE_LAUNCH(UPIPE_KIND_OPROJ_GEMM, launch_gemm(GK_OPROJ, m_ob[buf], m_wo, o, st));
  }
  // Host O complete when the caller's stream passes this point.
  if (o_host) UPIPE_CU(cudaStreamWaitEvent(st, cp->o_done[(s.nch - 1) % 3], 0));
  return UPIPE_OK;
}

// Layer backward; at most one of o_saved and o_host is non-null.
int layer_bwd(const upipe_cfg* cfg, const uint16_t* x, const uint16_t* Wqkv, const uint16_t* Wo,
              const uint16_t* dout, const float* lse, const uint16_t* o_saved, const uint16_t* o_host, uint16_t* dx,
              float* dWqkv, float* dWo, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  if (!check_cfg(cfg, true, &s)) return UPIPE_ERR_INVALID_ARG;
  if (!x || !Wqkv || !Wo || !dout || !lse || !dx || !dWqkv || !dWo || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dx) || !aligned16(dWqkv) || !aligned16(dWo) || !aligned16(ws) || (o_saved && !aligned16(o_saved)))
    return UPIPE_ERR_INVALID_ARG;
  const int o_mode = o_host ? kOHost : o_saved ? kODevice : kOWorkspace;
  const Plan pl = make_plan(s, 1, false, o_mode);
  if (ws_bytes < pl.total) return UPIPE_ERR_WS_TOO_SMALL;
  int* status = nullptr;
  if (int e = device_ready(&status)) return e;
  std::unique_lock<std::mutex> copy_lock;
  Copier* cp = nullptr;
  if (o_host) {
    copy_lock = std::unique_lock<std::mutex>(g_copier_mu);
    if (int e = copier(&cp)) return e;
  }
  const uint64_t limit = spin_limit_ns();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float2* rope = reinterpret_cast<float2*>(w + pl.off_rope);
  bf16* qkv = reinterpret_cast<bf16*>(w + pl.off_qkv);
  bf16* dO = reinterpret_cast<bf16*>(w + pl.off_dO);
  float* delta = reinterpret_cast<float*>(w + pl.off_delta);
  bf16* dqkv = reinterpret_cast<bf16*>(w + pl.off_dqkv);
  float* dkv_carry = reinterpret_cast<float*>(w + pl.off_dkv);
  float* carry = reinterpret_cast<float*>(w + pl.off_carry);
  const int64_t L = s.L;
  const int slots = s.U + 2 * s.kvc;
  const int m_tiles = static_cast<int>((L + 127) / 128);
  const int64_t Hd = static_cast<int64_t>(s.H) * 128;
  const float scale = static_cast<float>(1.0 / std::sqrt(128.0));
  const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(128.0));

  UPIPE_LAUNCH(UPIPE_KIND_ROPE_TABLE, launch_rope_table(rope, L, cfg->rope_theta, st));

  const bf16* obuf = o_saved ? reinterpret_cast<const bf16*>(o_saved) : reinterpret_cast<bf16*>(w + pl.off_o);
  const int64_t ld_o = o_saved ? Hd : static_cast<int64_t>(s.U) * 128;
  const size_t o_chunk_elems = static_cast<size_t>(L) * s.U * 128;
  CUtensorMap m_o1_mn;  // host mode: the second chunk buffer
  if (o_host) UPIPE_MAP(map2d(&m_o1_mn, obuf + o_chunk_elems, ld_o, L, ld_o, 64));
  CUtensorMap m_x, m_xmn, m_wqkv, m_wqkv_mn, m_qkv, m_wo_mn, m_dout, m_dout_mn, m_o_mn, m_do,
      m_dqkv_k, m_dqkv_mn;
  UPIPE_MAP(map2d(&m_x, x, s.D, L, s.D, 128));
  UPIPE_MAP(map2d(&m_xmn, x, s.D, L, s.D, 64));
  UPIPE_MAP(map2d(&m_wqkv, Wqkv, s.D, static_cast<uint64_t>(s.H + 2 * s.Hkv) * 128, s.D, 128));
  UPIPE_MAP(map2d(&m_wqkv_mn, Wqkv, s.D, static_cast<uint64_t>(s.H + 2 * s.Hkv) * 128, s.D, 64));
  UPIPE_MAP(map3d(&m_qkv, qkv, L, slots, 128, L * 128, 128));
  UPIPE_MAP(map2d(&m_wo_mn, Wo, Hd, s.D, Hd, 64));
  UPIPE_MAP(map2d(&m_dout, dout, s.D, L, s.D, 128));
  UPIPE_MAP(map2d(&m_dout_mn, dout, s.D, L, s.D, 64));
  UPIPE_MAP(map2d(&m_o_mn, obuf, ld_o, L, ld_o, 64));
  UPIPE_MAP(map3d(&m_do, dO, L, s.U, 128, L * 128, 128));
  UPIPE_MAP(map3d(&m_dqkv_k, dqkv, L, 2 * slots, 128, L * 128, 128));
  UPIPE_MAP(map3d(&m_dqkv_mn, dqkv, L, 2 * slots, 128, L * 128, 64));

  // Host mode: chunk c's O comes back into buffer c % 2.  The copy of
  // chunk c + 1 is issued once everything of chunk c - 1 (the last reader of
  // that buffer) is enqueued, and runs under chunk c's work.
  const bf16* oh = reinterpret_cast<const bf16*>(o_host);
  auto o_chunk = [&](int c) { return const_cast<bf16*>(obuf) + (c & 1) * o_chunk_elems; };
  if (o_host) {
    if (int e = copy_o_chunk(cp, o_chunk(0), oh, o_chunk_elems * 2, false, 0, st)) return e;
  }
  const int chunks_per_group = s.U < s.g ? s.g / s.U : 1;
  for (int c = 0; c < s.nch; ++c) {
    const Chunk ch = chunk_of(s, c);
    const int cg = c % chunks_per_group;
    const bool group_first = cg == 0;
    const bool group_last = cg == chunks_per_group - 1;
    const bool emit_kv = group_last;  // K/V gradients complete for this chunk's KV heads
    if (o_host && c + 1 < s.nch) {
      if (int e = copy_o_chunk(cp, o_chunk(c + 1), oh + (c + 1) * o_chunk_elems, o_chunk_elems * 2, false,
                               (c + 1) & 1, st))
        return e;
    }

    // Recompute Q/K/V of the chunk (a-1, a-2).
    GemmParams g = gemm_base(status, limit);
    g.M = static_cast<int>(L);
    g.N = slots * 128;
    g.K = s.D;
    g.m_tiles = m_tiles;
    g.n_tiles = slots;
    g.k_blocks = s.D / 64;
    g.L = static_cast<int>(L);
    for (int sl = 0; sl < slots; ++sl) g.tab0[sl] = static_cast<int16_t>(w_block(s, ch, sl));
    g.out = qkv;
    g.rope_slots = s.U + s.kvc;
    g.rope = rope;
    UPIPE_LAUNCH(UPIPE_KIND_QKV_GEMM, launch_gemm(GK_QKV, m_x, m_wqkv, g, st));

    // Recompute O_c unless the caller kept it (a-3), from the forward's LSE:
    // the probabilities are final at once, and are the ones the backward
    // kernels use.
    if (!o_saved && !o_host) {
      AttnFwdParams a;
      std::memset(&a, 0, sizeof(a));
      a.mode = kLseIn;
      a.lse_in = lse + static_cast<int64_t>(ch.q0) * L;
      a.L = static_cast<int>(L);
      a.nheads = s.U;
      a.g_loc = s.U / s.kvc;
      a.k_z0 = s.U;
      a.v_z0 = s.U + s.kvc;
      a.o = const_cast<bf16*>(obuf);
      a.o_row = ld_o;
      a.o_head = 128;
      a.lse = nullptr;
      a.write_lse = 0;
      a.scale_log2 = scale_log2;
      a.status = status;
      a.limit_ns = limit;
      UPIPE_LAUNCH(UPIPE_KIND_ATTN_FWD, launch_attn_fwd(m_qkv, m_qkv, m_qkv, a, m_tiles, st));
    }
    const int o_col0 = o_saved ? ch.q0 * 128 : 0;
    const bf16* o_rows = o_host ? o_chunk(c) : obuf + o_col0;
    if (o_host) UPIPE_CU(cudaStreamWaitEvent(st, cp->o_done[c & 1], 0));  // O_c is back

    // dO_c = dout Wo[:, cols_c], and Delta = rowsum(dO_c * O_c).
    GemmParams d = gemm_base(status, limit);
    d.M = static_cast<int>(L);
    d.N = s.U * 128;
    d.K = s.D;
    d.m_tiles = m_tiles;
    d.n_tiles = s.U;
    d.k_blocks = s.D / 64;
    d.b_col0 = ch.q0 * 128;
    d.L = static_cast<int>(L);
    d.out = dO;
    d.o_rows = o_rows;
    d.ld_o = ld_o;
    d.lse_in = lse + static_cast<int64_t>(ch.q0) * L;
    d.ld_rec = delta;
    UPIPE_LAUNCH(UPIPE_KIND_DO_GEMM, launch_gemm(GK_DO, m_dout, m_wo_mn, d, st));

    // dWo[:, cols_c] = dout^T O_c.
    GemmParams dw = gemm_base(status, limit);
    dw.M = s.D;
    dw.N = s.U * 128;
    dw.K = static_cast<int>(L);
    dw.m_tiles = s.D / 128;
    dw.n_tiles = s.U;
    dw.k_blocks = static_cast<int>((L + 63) / 64);
    dw.b_col0 = o_col0;
    dw.out_col0 = ch.q0 * 128;
    dw.out = dWo;
    dw.ld_out = Hd;
    // K (tokens) in two halves reduced into the zeroed columns, split where
    // dWqkv splits (depends on L alone).
    dw.k_mid = dw.k_blocks >= 2 && dw.m_tiles <= kMaxSlots ? (dw.k_blocks + 1) / 2 : 0;
    if (dw.k_mid > 0) {
      int16_t rows[kMaxSlots];
      for (int b = 0; b < dw.m_tiles; ++b) rows[b] = static_cast<int16_t>(b);
      UPIPE_LAUNCH(UPIPE_KIND_ZERO_ROWS,
                   launch_zero_rows(dWo + dw.out_col0, Hd, dw.N, rows, dw.m_tiles, st));
    }
    UPIPE_LAUNCH(UPIPE_KIND_DWO_GEMM,
                 launch_gemm(GK_DWO, m_dout_mn, o_host && (c & 1) ? m_o1_mn : m_o_mn, dw, st));

    // Attention backward (a-5): dQ, then dK/dV (carried when U < g).
    AttnBwdParams b;
    std::memset(&b, 0, sizeof(b));
    b.L = static_cast<int>(L);
    b.nheads = s.U;
    b.g_loc = s.U / s.kvc;
    b.nkv = s.kvc;
    b.q_z0 = 0;
    b.k_z0 = s.U;
    b.v_z0 = s.U + s.kvc;
    b.do_z0 = 0;
    b.ld = delta;
    b.scale = scale;
    b.scale_log2 = scale_log2;
    b.dq = dqkv;
    b.dq_row = 128;
    b.dq_head = L * 128;
    b.dk = dqkv + static_cast<int64_t>(s.U) * L * 128;
    b.dv = dqkv + static_cast<int64_t>(s.U + s.kvc) * L * 128;
    b.dkv_row = 128;
    b.dkv_head = L * 128;
    b.lo_off = static_cast<int64_t>(slots) * L * 128;
    b.dkv_carry = dkv_carry;
    b.carry_in = !group_first;
    b.carry_out = !group_last;
    b.rope = rope;
    b.status = status;
    b.limit_ns = limit;
    if (int e = launch_attn_bwd_pair(m_qkv, m_qkv, m_qkv, m_do, b, m_tiles, st)) return e;

    // dWqkv rows of the chunk: q slots always, k/v slots once complete.
    const int out_slots = emit_kv ? slots : s.U;
    GemmParams wq = gemm_base(status, limit);
    wq.M = out_slots * 128;
    wq.N = s.D;
    wq.K = static_cast<int>(L);
    wq.m_tiles = out_slots;
    wq.n_tiles = s.D / 128;
    wq.k_blocks = static_cast<int>((L + 63) / 64);
    for (int sl = 0; sl < out_slots; ++sl) {
      wq.tab0[sl] = static_cast<int16_t>(sl);
      wq.tab1[sl] = static_cast<int16_t>(w_block(s, ch, sl));
    }
    wq.out = dWqkv;
    wq.ld_out = s.D;
    wq.lo_z = slots;
    // K (tokens) in two halves reduced into zeroed rows; the split point
    // depends on L alone.
    wq.k_mid = wq.k_blocks >= 2 ? (wq.k_blocks + 1) / 2 : 0;
    if (wq.k_mid > 0)
      UPIPE_LAUNCH(UPIPE_KIND_ZERO_ROWS, launch_zero_rows(dWqkv, s.D, s.D, wq.tab1, out_slots, st));
    UPIPE_LAUNCH(UPIPE_KIND_DWQKV_GEMM, launch_gemm(GK_DWQKV, m_dqkv_mn, m_xmn, wq, st));

    // dx32 (+)= dqkv_c W_c, K slots in the canonical order: per KV group,
    // its query heads ascending, then its k and v rows.
    GemmParams dxp = gemm_base(status, limit);
    int ks = 0;
    const int gl = s.U / s.kvc;  // query heads per KV head within the chunk
    for (int j = 0; j < s.kvc; ++j) {
      for (int t = 0; t < gl; ++t) {
        const int sl = j * gl + t;
        dxp.tab0[ks] = static_cast<int16_t>(sl);
        dxp.tab1[ks] = static_cast<int16_t>(w_block(s, ch, sl));
        ++ks;
      }
      if (emit_kv) {
        for (int sl : {s.U + j, s.U + s.kvc + j}) {
          dxp.tab0[ks] = static_cast<int16_t>(sl);
          dxp.tab1[ks] = static_cast<int16_t>(w_block(s, ch, sl));
          ++ks;
        }
      }
    }
    dxp.M = static_cast<int>(L);
    dxp.N = s.D;
    dxp.K = ks * 128;
    dxp.m_tiles = m_tiles;
    dxp.n_tiles = s.D / 128;
    dxp.k_blocks = ks * 2;
    dxp.out = dx;
    dxp.ld_out = s.D;
    dxp.carry = carry;
    dxp.lo_z = slots;
    dxp.carry_in = c > 0;
    dxp.final_out = c == s.nch - 1;
    UPIPE_LAUNCH(UPIPE_KIND_DX_GEMM, launch_gemm(GK_DX, m_dqkv_k, m_wqkv_mn, dxp, st));
  }
  return UPIPE_OK;
}

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" {

size_t upipe_workspace_bytes(const upipe_cfg* cfg, int pass, int core_only, int o_mode) {
  Shape s;
  if ((pass != 0 && pass != 1) || o_mode < 0 || o_mode > 2 || !check_cfg(cfg, !core_only, &s)) return 0;
  return make_plan(s, pass, core_only != 0, o_mode).total;
}

int upipe_activation_bytes(const upipe_cfg* cfg, int pass, int core_only, int o_mode, size_t* chunk_bytes,
                           size_t* fixed_bytes) {
  Shape s;
  if ((pass != 0 && pass != 1) || o_mode < 0 || o_mode > 2 || !check_cfg(cfg, !core_only, &s))
    return UPIPE_ERR_INVALID_ARG;
  const Plan p = make_plan(s, pass, core_only != 0, o_mode);
  if (chunk_bytes) *chunk_bytes = p.chunk_bytes();
  if (fixed_bytes) *fixed_bytes = p.fixed_bytes();
  return UPIPE_OK;
}

int upipe_choose_u(const upipe_cfg* cfg, size_t budget_bytes, int pass, int core_only, int o_mode) {
  if (!cfg || pass < 0 || pass > 2 || o_mode < 0 || o_mode > 2) return UPIPE_ERR_INVALID_ARG;
  upipe_cfg c = *cfg;
  Shape s;
  c.U = c.H;  // U = H is valid whenever the rest of the configuration is
  if (!check_cfg(&c, !core_only, &s)) return UPIPE_ERR_INVALID_ARG;
  for (int u = c.H; u >= 1; --u) {
    c.U = u;
    if (!check_cfg(&c, !core_only, &s)) continue;
    size_t need = 0;
    for (int ps = 0; ps < 2; ++ps)
      if (pass == 2 || pass == ps) {
        const size_t b = make_plan(s, ps, core_only != 0, o_mode).total;
        need = b > need ? b : need;
      }
    if (need <= budget_bytes) return u;
  }
  return UPIPE_ERR_WS_TOO_SMALL;
}

int upipe_attn_fwd(const upipe_cfg* cfg, const uint16_t* x, const uint16_t* Wqkv, const uint16_t* Wo, uint16_t* out,
                   float* lse, uint16_t* o_saved, void* ws, size_t ws_bytes, void* stream) {
  return layer_fwd(cfg, x, Wqkv, Wo, out, lse, o_saved, nullptr, ws, ws_bytes, stream);
}

int upipe_attn_bwd(const upipe_cfg* cfg, const uint16_t* x, const uint16_t* Wqkv, const uint16_t* Wo,
                   const uint16_t* dout, const float* lse, const uint16_t* o_saved, uint16_t* dx, float* dWqkv,
                   float* dWo, void* ws, size_t ws_bytes, void* stream) {
  return layer_bwd(cfg, x, Wqkv, Wo, dout, lse, o_saved, nullptr, dx, dWqkv, dWo, ws, ws_bytes, stream);
}

int upipe_attn_fwd_host_o(const upipe_cfg* cfg, const uint16_t* x, const uint16_t* Wqkv, const uint16_t* Wo,
                          uint16_t* out, float* lse, uint16_t* o_host, void* ws, size_t ws_bytes, void* stream) {
  if (!o_host || !host_pinned(o_host)) return UPIPE_ERR_INVALID_ARG;
  return layer_fwd(cfg, x, Wqkv, Wo, out, lse, nullptr, o_host, ws, ws_bytes, stream);
}

int upipe_attn_bwd_host_o(const upipe_cfg* cfg, const uint16_t* x, const uint16_t* Wqkv, const uint16_t* Wo,
                          const uint16_t* dout, const float* lse, const uint16_t* o_host, uint16_t* dx, float* dWqkv,
                          float* dWo, void* ws, size_t ws_bytes, void* stream) {
  if (!o_host || !host_pinned(o_host)) return UPIPE_ERR_INVALID_ARG;
  return layer_bwd(cfg, x, Wqkv, Wo, dout, lse, nullptr, o_host, dx, dWqkv, dWo, ws, ws_bytes, stream);
}

int upipe_attn_core_fwd(const upipe_cfg* cfg, const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                        float* lse, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  if (!check_cfg(cfg, false, &s)) return UPIPE_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return UPIPE_ERR_INVALID_ARG;
  (void)ws;
  (void)ws_bytes;
  int* status = nullptr;
  if (int e = device_ready(&status)) return e;
  const uint64_t limit = spin_limit_ns();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t L = s.L;
  const int m_tiles = static_cast<int>((L + 127) / 128);
  const int64_t Hd = static_cast<int64_t>(s.H) * 128, Hkvd = static_cast<int64_t>(s.Hkv) * 128;
  CUtensorMap mq, mk, mv;
  UPIPE_MAP(map3d(&mq, q, L, s.H, Hd, 128, 128));
  UPIPE_MAP(map3d(&mk, k, L, s.Hkv, Hkvd, 128, 128));
  UPIPE_MAP(map3d(&mv, v, L, s.Hkv, Hkvd, 128, 128));
  for (int c = 0; c < s.nch; ++c) {
    const Chunk ch = chunk_of(s, c);
    AttnFwdParams a;
    std::memset(&a, 0, sizeof(a));
    a.L = static_cast<int>(L);
    a.nheads = s.U;
    a.g_loc = s.U / s.kvc;
    a.q_z0 = ch.q0;
    a.k_z0 = ch.kv0;
    a.v_z0 = ch.kv0;
    a.o = reinterpret_cast<bf16*>(o) + static_cast<int64_t>(ch.q0) * 128;
    a.o_row = Hd;
    a.o_head = 128;
    a.lse = lse + static_cast<int64_t>(ch.q0) * L;
    a.write_lse = 1;
    a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(128.0));
    a.status = status;
    a.limit_ns = limit;
    UPIPE_LAUNCH(UPIPE_KIND_ATTN_FWD, launch_attn_fwd(mq, mk, mv, a, m_tiles, st));
  }
  return UPIPE_OK;
}

int upipe_attn_core_bwd(const upipe_cfg* cfg, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const uint16_t* o, const float* lse, const uint16_t* dout_o, uint16_t* dq, uint16_t* dk,
                        uint16_t* dv, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  if (!check_cfg(cfg, false, &s)) return UPIPE_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse || !dout_o || !dq || !dk || !dv || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout_o) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(ws))
    return UPIPE_ERR_INVALID_ARG;
  const Plan pl = make_plan(s, 1, true, false);
  if (ws_bytes < pl.total) return UPIPE_ERR_WS_TOO_SMALL;
  int* status = nullptr;
  if (int e = device_ready(&status)) return e;
  const uint64_t limit = spin_limit_ns();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* delta = reinterpret_cast<float*>(w + pl.off_delta);
  float* dkv_carry = reinterpret_cast<float*>(w + pl.off_dkv);
  const int64_t L = s.L;
  const int m_tiles = static_cast<int>((L + 127) / 128);
  const int64_t Hd = static_cast<int64_t>(s.H) * 128, Hkvd = static_cast<int64_t>(s.Hkv) * 128;
  CUtensorMap mq, mk, mv, mdo;
  UPIPE_MAP(map3d(&mq, q, L, s.H, Hd, 128, 128));
  UPIPE_MAP(map3d(&mk, k, L, s.Hkv, Hkvd, 128, 128));
  UPIPE_MAP(map3d(&mv, v, L, s.Hkv, Hkvd, 128, 128));
  UPIPE_MAP(map3d(&mdo, dout_o, L, s.H, Hd, 128, 128));
  const int chunks_per_group = s.U < s.g ? s.g / s.U : 1;
  for (int c = 0; c < s.nch; ++c) {
    const Chunk ch = chunk_of(s, c);
    const int cg = c % chunks_per_group;
    UPIPE_LAUNCH(UPIPE_KIND_DELTA, launch_delta(reinterpret_cast<const bf16*>(o) + static_cast<int64_t>(ch.q0) * 128, Hd, 128,
                          reinterpret_cast<const bf16*>(dout_o) + static_cast<int64_t>(ch.q0) * 128, Hd, 128,
                          lse + static_cast<int64_t>(ch.q0) * L, delta, L, s.U, st));
    AttnBwdParams b;
    std::memset(&b, 0, sizeof(b));
    b.L = static_cast<int>(L);
    b.nheads = s.U;
    b.g_loc = s.U / s.kvc;
    b.nkv = s.kvc;
    b.q_z0 = ch.q0;
    b.k_z0 = ch.kv0;
    b.v_z0 = ch.kv0;
    b.do_z0 = ch.q0;
    b.ld = delta;
    b.scale = static_cast<float>(1.0 / std::sqrt(128.0));
    b.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(128.0));
    b.dq = reinterpret_cast<bf16*>(dq) + static_cast<int64_t>(ch.q0) * 128;
    b.dq_row = Hd;
    b.dq_head = 128;
    b.dk = reinterpret_cast<bf16*>(dk) + static_cast<int64_t>(ch.kv0) * 128;
    b.dv = reinterpret_cast<bf16*>(dv) + static_cast<int64_t>(ch.kv0) * 128;
    b.dkv_row = Hkvd;
    b.dkv_head = 128;
    b.dkv_carry = dkv_carry;
    b.carry_in = cg != 0;
    b.carry_out = cg != chunks_per_group - 1;
    b.rope = nullptr;
    b.status = status;
    b.limit_ns = limit;
    if (int e = launch_attn_bwd_pair(mq, mk, mv, mdo, b, m_tiles, st)) return e;
  }
  return UPIPE_OK;
}

int upipe_offload_async(void* host_dst, const void* dev_src, size_t bytes, void* stream) {
  return async_copy(host_dst, dev_src, bytes, true, static_cast<cudaStream_t>(stream));
}

int upipe_prefetch_async(void* dev_dst, const void* host_src, size_t bytes, void* stream) {
  return async_copy(dev_dst, host_src, bytes, false, static_cast<cudaStream_t>(stream));
}

int upipe_copies_join(void* stream) {
  std::lock_guard<std::mutex> lock(g_copier_mu);
  Copier* c = nullptr;
  if (int e = copier(&c)) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaEventRecord(c->done_d2h, c->d2h) != cudaSuccess || cudaEventRecord(c->done_h2d, c->h2d) != cudaSuccess ||
      cudaStreamWaitEvent(st, c->done_d2h, 0) != cudaSuccess || cudaStreamWaitEvent(st, c->done_h2d, 0) != cudaSuccess)
    return UPIPE_ERR_CUDA;
  return UPIPE_OK;
}

int upipe_last_device_status(void* stream) {
  int* status = nullptr;
  if (int e = device_ready(&status)) return e;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return UPIPE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return UPIPE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return UPIPE_ERR_CUDA;
  return v ? UPIPE_ERR_DEVICE_TIMEOUT : UPIPE_OK;
}

int upipe_debug_wait_timeout(uint64_t limit_ns, void* stream) {
  int* status = nullptr;
  if (int e = device_ready(&status)) return e;
  return launch_wait_selftest(status, limit_ns, static_cast<cudaStream_t>(stream)) == cudaSuccess ? UPIPE_OK
                                                                                                   : UPIPE_ERR_CUDA;
}

int64_t upipe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void upipe_profile_enable(int on) { g_profile.store(on != 0, std::memory_order_relaxed); }

int upipe_profile_read(double* ms, int64_t* launches, int n) {
  for (int k = 0; k < n; ++k) {
    if (ms) ms[k] = 0.0;
    if (launches) launches[k] = 0;
  }
  for (const ProfRec& r : g_prof) {
    cudaEventSynchronize(r.b);
    float t = 0.f;
    cudaEventElapsedTime(&t, r.a, r.b);
    if (r.kind < n) {
      if (ms) ms[r.kind] += t;
      if (launches) launches[r.kind] += 1;
    }
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof.clear();
  return UPIPE_KIND_COUNT;
}

const char* upipe_strerror(int code) {
  switch (code) {
    case UPIPE_OK: return "ok";
    case UPIPE_ERR_INVALID_ARG: return "invalid argument (shape, null or misaligned pointer)";
    case UPIPE_ERR_WS_TOO_SMALL: return "workspace too small";
    case UPIPE_ERR_CUDA: return "CUDA error";
    case UPIPE_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
    case UPIPE_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103 (GB300)";
    case UPIPE_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the no-allocation entry point holds";
  }
  return "unknown error";
}

}  // extern "C"
