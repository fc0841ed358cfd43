// flint_moe_route_noalloc: routing with the library's own fixed scratch
// (declared in include/flint_moe.h).  Same kernel and numerics as
// flint_moe_route; only where the intermediates live differs.
#include <mutex>

#include <cuda_runtime.h>
#include <stdint.h>

#include "flint_moe.h"
#include "internal.h"

namespace flint {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB per device

// The scratch itself: zero at module load, like all static device memory.
__device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

// Device addresses of the scratch, one per CUDA context that has called the
// entry point, keyed by the context's process-unique id (cuCtxGetId): a
// context created later (another device, a driver-API context, or the primary
// context re-created after cudaDeviceReset) never matches an older entry.
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
constexpr int kMaxContexts = 64;
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxContexts];
int g_scratch_n = 0;

using CtxGetCurrentFn = int (*)(void**);
using CtxGetIdFn = int (*)(void*, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

struct NoAllocLayout {
  size_t tok_cnt, logits, ids, tw, total;
};

// Regions the router kernel touches when it builds no expert grouping: the
// per-token-block counters (must be zero at launch), the bf16 logits and the
// kernel's own copies of ids / tw.
NoAllocLayout noalloc_layout(const flint_moe_shape& s) {
  NoAllocLayout L{};
  const size_t M = s.M, E = s.E, k = s.top_k;
  L.tok_cnt = 0;
  L.logits = round256(4 * ((M + kRouteTokens - 1) / kRouteTokens));
  L.ids = L.logits + round256(2 * M * E);
  L.tw = L.ids + round256(4 * M * k);
  L.total = L.tw + round256(4 * M * k);
  return L;
}

// Well-formed (H a multiple of 64, as for flint_moe_route); the kernel runs
// H in whole 128-wide slices.
bool shape_ok(const flint_moe_shape* s) {
  if (!s) return false;
  if (s->M < 0 || s->H < 64 || s->H % 64 != 0) return false;
  if (s->E < 1 || s->E > kMaxE) return false;
  if (s->top_k < 1 || s->top_k > s->E || s->top_k > kMaxTopK) return false;
  return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Id of the calling thread's current CUDA context (0 when it has none yet).
// The driver entry points are looked up through the runtime (no link against
// the driver library).
int current_context_id(unsigned long long* id) {
  if (!g_ctx_get_current || !g_ctx_get_id) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || !f1)
      return FLINT_ERR_CUDA;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess || !f2)
      return FLINT_ERR_CUDA;
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
  }
  void* ctx = nullptr;
  if (g_ctx_get_current(&ctx) != 0) return FLINT_ERR_CUDA;
  *id = 0;
  if (ctx && g_ctx_get_id(ctx, id) != 0) return FLINT_ERR_CUDA;
  return FLINT_OK;
}

// Device address of the scratch in the current context.  The first call in
// a context looks it up with cudaGetSymbolAddress (which may load the module
// into that context, so it belongs outside stream capture); later calls in
// the same context reuse the cached address.
int scratch_address(void** out) {
  unsigned long long id = 0;
  int rc = current_context_id(&id);
  if (rc != FLINT_OK) return rc;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (id != 0)
    for (int i = 0; i < g_scratch_n; ++i)
      if (g_scratch[i].ctx_id == id) {
        *out = g_scratch[i].addr;
        return FLINT_OK;
      }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return FLINT_ERR_CUDA;
  if (id == 0) {  // the lookup above made the runtime's context current
    rc = current_context_id(&id);
    if (rc != FLINT_OK) return rc;
  }
  if (id != 0) {
    if (g_scratch_n < kMaxContexts) {
      g_scratch[g_scratch_n++] = {id, p};
    } else {  // more contexts than slots: recycle the oldest entry
      for (int i = 1; i < kMaxContexts; ++i) g_scratch[i - 1] = g_scratch[i];
      g_scratch[kMaxContexts - 1] = {id, p};
    }
  }
  *out = p;
  return FLINT_OK;
}

}  // namespace
}  // namespace flint

using namespace flint;

extern "C" {

size_t flint_moe_route_noalloc_bytes(const flint_moe_shape* shape) {
  if (!shape_ok(shape) || shape->H % 128 != 0) return 0;
  return noalloc_layout(*shape).total;
}

size_t flint_moe_route_noalloc_capacity(void) { return kNoAllocScratchBytes; }

int flint_moe_route_noalloc(const void* x, const void* router_w, const flint_moe_shape* shape,
                            int32_t* ids, float* tw, flint_stream_t stream) {
  if (!shape_ok(shape)) return FLINT_ERR_INVALID_ARG;
  if (shape->H % 128 != 0) return FLINT_ERR_UNSUPPORTED;
  if (shape->M == 0) return FLINT_OK;  // an empty batch: nothing to launch
  if (!x || !router_w || !ids || !tw) return FLINT_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(router_w, 16) || !aligned(ids, 4) || !aligned(tw, 4))
    return FLINT_ERR_INVALID_ARG;
  const NoAllocLayout L = noalloc_layout(*shape);
  if (L.total > kNoAllocScratchBytes) return FLINT_ERR_SCRATCH;

  void* base = nullptr;
  const int rc = scratch_address(&base);
  if (rc != FLINT_OK) return rc;
  char* b = static_cast<char*>(base);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the counters must read zero at launch; the kernel also leaves them at
  // zero, the clear only guards against an earlier launch that did not finish
  if (cudaMemsetAsync(b + L.tok_cnt, 0, L.logits - L.tok_cnt, st) != cudaSuccess)
    return FLINT_ERR_CUDA;

  MoEArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.router_w = static_cast<const uint16_t*>(router_w);
  a.ids_out = ids;
  a.tw_out = tw;
  a.M = shape->M; a.H = shape->H; a.E = shape->E; a.k = shape->top_k;
  a.I = 128; a.SI = 0;
  a.ws.tok_cnt = reinterpret_cast<int*>(b + L.tok_cnt);
  a.ws.logits = reinterpret_cast<uint16_t*>(b + L.logits);
  a.ws.ids = reinterpret_cast<int*>(b + L.ids);
  a.ws.tw = reinterpret_cast<float*>(b + L.tw);
  if (launch_route(a, false, st, false) != cudaSuccess) return FLINT_ERR_CUDA;
  return FLINT_OK;
}

}  // extern "C"
