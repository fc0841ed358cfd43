// flint_moe_route_noalloc: routing with the library's own fixed scratch
// (declared in include/flint_moe.h).  Same kernel and numerics as
// flint_moe_route; only where the intermediates live differs.
#include <atomic>

#include <cuda_runtime.h>
#include <stdint.h>

#include "flint_moe.h"
#include "internal.h"

namespace flint {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB per device
constexpr int kMaxDevices = 64;

// The scratch itself: zero at module load, like all static device memory.
__device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

std::atomic<void*> g_scratch_addr[kMaxDevices];

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

bool shape_ok(const flint_moe_shape* s) {
  if (!s) return false;
  if (s->M < 0 || s->H < 128 || s->H % 128 != 0) return false;
  if (s->E < 1 || s->E > kMaxE) return false;
  if (s->top_k < 1 || s->top_k > s->E || s->top_k > kMaxTopK) return false;
  return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device address of this device's copy of the scratch, looked up once per
// device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLINT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FLINT_ERR_UNSUPPORTED;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return FLINT_ERR_CUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return FLINT_OK;
}

}  // namespace
}  // namespace flint

using namespace flint;

extern "C" {

size_t flint_moe_route_noalloc_bytes(const flint_moe_shape* shape) {
  if (!shape_ok(shape)) return 0;
  return noalloc_layout(*shape).total;
}

size_t flint_moe_route_noalloc_capacity(void) { return kNoAllocScratchBytes; }

int flint_moe_route_noalloc(const void* x, const void* router_w, const flint_moe_shape* shape,
                            int32_t* ids, float* tw, flint_stream_t stream) {
  if (!shape_ok(shape)) return FLINT_ERR_INVALID_ARG;
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
