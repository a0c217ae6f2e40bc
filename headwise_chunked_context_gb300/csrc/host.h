// Host-side helpers shared by the entry-point files (upipe.cu for the
// attention layer, alst.cu for the sequence-tiled MLP and loss): argument
// checks, device readiness, TMA tensor maps and launch accounting.  Defined
// in upipe.cu.
#pragma once

#include <atomic>
#include <cstring>
#include <vector>

#include "upipe.h"
#include "upipe_internal.h"

namespace upipe {

bool aligned16(const void* p);
// Bound of every device-side wait (UPIPE_SPIN_LIMIT_NS, default 2 s).
uint64_t spin_limit_ns();
// Checks that the current device is an sm_103 part and returns the address
// of its status word; UPIPE_OK or an error code.
int device_ready(int** status);
// bf16 [rows, cols] with leading dimension ld (elements); box 64 x box_rows,
// 128-byte swizzle.
bool map2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_rows);
// bf16 heads of 128: element (c, row, head) at base + row*row_stride + head*head_stride.
bool map3d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t heads, uint64_t row_stride,
           uint64_t head_stride, uint32_t box_rows);

// Launch accounting: a counter of every kernel launch, and optional CUDA
// event pairs recorded around each launch on the launching stream.
struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};
extern std::atomic<int64_t> g_launches;
extern std::atomic<bool> g_profile;
extern thread_local bool t_no_profile;
extern std::vector<ProfRec> g_prof;
cudaEvent_t pool_event();

template <class F>
cudaError_t counted(int kind, cudaStream_t st, F&& launch) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_profile.load(std::memory_order_relaxed) || t_no_profile) return launch();
  ProfRec r{kind, pool_event(), pool_event()};
  cudaEventRecord(r.a, st);
  const cudaError_t e = launch();
  cudaEventRecord(r.b, st);
  g_prof.push_back(r);
  return e;
}

inline GemmParams gemm_base(int* status, uint64_t limit) {
  GemmParams g;
  std::memset(&g, 0, sizeof(g));
  g.status = status;
  g.limit_ns = limit;
  return g;
}

}  // namespace upipe

#define UPIPE_CU(x)                                \
  do {                                             \
    if ((x) != cudaSuccess) return UPIPE_ERR_CUDA; \
  } while (0)
// Launch expression x on stream `st` (a local of the caller), counted.
#define UPIPE_LAUNCH(kind, x) UPIPE_CU(::upipe::counted(kind, st, [&] { return (x); }))
#define UPIPE_MAP(x)                 \
  do {                               \
    if (!(x)) return UPIPE_ERR_CUDA; \
  } while (0)
