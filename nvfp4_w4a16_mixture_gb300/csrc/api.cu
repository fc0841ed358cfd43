// C-ABI entry points of libflint_moe (declared in include/flint_moe.h).
#include <atomic>

#include <cuda_runtime.h>
#include <stdint.h>

#include "flint_moe.h"
#include "internal.h"

namespace flint {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static std::atomic<int> g_fault_site{0};  // test hook, see flint_moe_debug_fault
static std::atomic<int> g_prefer{0};      // flint_moe_prefer_path
int debug_fault_site() { return g_fault_site.load(std::memory_order_relaxed); }

// A well-formed shape: H, I and SI multiples of 64 (the unit of the block's
// interface), counts in range.
static bool shape_valid(const flint_moe_shape* s) {
  if (!s) return false;
  if (s->M < 0 || s->H < 64 || s->H % 64 != 0) return false;
  if (s->E < 1 || s->E > kMaxE) return false;
  if (s->top_k < 1 || s->top_k > s->E || s->top_k > kMaxTopK) return false;
  if (s->I < 64 || s->I % 64 != 0) return false;
  if (s->SI < 0 || s->SI % 64 != 0) return false;
  // element counts addressed with 32-bit indices in places
  if ((int64_t)s->M * s->top_k > (int64_t)1 << 30) return false;
  if ((int64_t)s->H * 2 * s->I > (int64_t)1 << 31) return false;
  return true;
}

// Shapes the kernels run: every K extent a whole number of 128-wide slices.
static bool shape_supported(const flint_moe_shape* s) {
  return s->H % 128 == 0 && s->I % 128 == 0 && s->SI % 128 == 0;
}

// The path flint_moe_forward takes for a valid, supported shape with M > 0.
// The three-kernel decode path is the default for few tokens (it measures
// faster than the single launch at every M it serves); the single launch
// runs where the caller prefers it and it supports the shape.
static int plan(const flint_moe_shape& s, int sms) {
  if (s.M > kDecodeMaxTokens && grouped_supported(s)) return FLINT_PATH_GROUPED;
  if (g_prefer.load(std::memory_order_relaxed) == FLINT_PATH_SINGLE_LAUNCH && fused_supported(s, sms))
    return FLINT_PATH_SINGLE_LAUNCH;
  if (decode2_supported(s)) return FLINT_PATH_DECODE;
  if (fused_supported(s, sms)) return FLINT_PATH_SINGLE_LAUNCH;
  return FLINT_PATH_DECODE_FALLBACK;
}

WsLayout ws_layout(const flint_moe_shape& s) {
  WsLayout L{};
  const size_t M = s.M, H = s.H, E = s.E, k = s.top_k, I = s.I, SI = s.SI;
  const size_t np = M * k;
  const size_t nchunks = (np + 1023) / 1024;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.status = take(16);
  L.glob_cnt = take(16);
  L.fd_cnt = take(16);
  L.hblk_cnt = take(4 * (H / 16));
  L.tok_cnt = take(4 * ((M + kRouteTokens - 1) / kRouteTokens));
  L.logits = take(2 * M * E);
  L.ids = take(4 * np);
  L.tw = take(4 * np);
  L.e_cnt = take(4 * E);
  L.e_off = take(4 * (E + 1));
  L.uniq = take(4 * (E + 1));
  L.sorted_pairs = take(4 * np);
  L.rowof = take(4 * np);
  L.urec = take(4 * (size_t)kUrecInts * (np < E ? np : E));
  L.gcnt = take(4 * 2 * nchunks * E);
  L.act = take(2 * np * I);
  L.sact = take(2 * M * (SI > 0 ? SI : 1));
  L.y = take(2 * np * H);
  L.ys = take(2 * M * H);
  const bool grouped = M > (size_t)kDecodeMaxTokens;
  L.x_perm = take(grouped ? 2 * np * H : 16);
  L.st_table = take(grouped ? 16 * grouped_st_entries(s) : 16);
  L.st_count = take(16);
  L.x16 = take(M <= (size_t)kX16MaxTokens ? 2 * M * H : 16);
  L.x16_exp = take(4 * M);
  L.xn = take(2 * M * H);
  L.total = off;
  return L;
}

Ws ws_pointers(void* base, const WsLayout& L) {
  char* b = static_cast<char*>(base);
  Ws w;
  w.status = reinterpret_cast<int*>(b + L.status);
  w.fd_cnt = reinterpret_cast<int*>(b + L.fd_cnt);
  w.tok_cnt = reinterpret_cast<int*>(b + L.tok_cnt);
  w.glob_cnt = reinterpret_cast<int*>(b + L.glob_cnt);
  w.hblk_cnt = reinterpret_cast<int*>(b + L.hblk_cnt);
  w.logits = reinterpret_cast<uint16_t*>(b + L.logits);
  w.ids = reinterpret_cast<int*>(b + L.ids);
  w.tw = reinterpret_cast<float*>(b + L.tw);
  w.e_cnt = reinterpret_cast<int*>(b + L.e_cnt);
  w.e_off = reinterpret_cast<int*>(b + L.e_off);
  w.uniq = reinterpret_cast<int*>(b + L.uniq);
  w.sorted_pairs = reinterpret_cast<int*>(b + L.sorted_pairs);
  w.rowof = reinterpret_cast<int*>(b + L.rowof);
  w.urec = reinterpret_cast<int*>(b + L.urec);
  w.gcnt = reinterpret_cast<int*>(b + L.gcnt);
  w.act = reinterpret_cast<uint16_t*>(b + L.act);
  w.x16 = reinterpret_cast<uint16_t*>(b + L.x16);
  w.x16_exp = reinterpret_cast<int*>(b + L.x16_exp);
  w.xn = reinterpret_cast<uint16_t*>(b + L.xn);
  w.sact = reinterpret_cast<uint16_t*>(b + L.sact);
  w.y = reinterpret_cast<uint16_t*>(b + L.y);
  w.ys = reinterpret_cast<uint16_t*>(b + L.ys);
  w.x_perm = reinterpret_cast<uint16_t*>(b + L.x_perm);
  w.st_table = reinterpret_cast<int*>(b + L.st_table);
  w.st_count = reinterpret_cast<int*>(b + L.st_count);
  return w;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Streaming multiprocessors of the current device (cached per device).
static cudaError_t device_sms(int* sms) {
  static std::atomic<int> cache[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    err = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  *sms = v;
  return cudaSuccess;
}

}  // namespace flint

using namespace flint;

extern "C" {

size_t flint_moe_workspace_bytes(const flint_moe_shape* shape) {
  if (!shape_valid(shape) || !shape_supported(shape)) return 0;
  return ws_layout(*shape).total;
}

int flint_moe_route(const void* x, const void* router_w, const flint_moe_shape* shape, int32_t* ids,
                    float* tw, void* workspace, size_t workspace_bytes, flint_stream_t stream) {
  if (!shape_valid(shape)) return FLINT_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return FLINT_ERR_UNSUPPORTED;
  if (shape->M == 0) return FLINT_OK;  // an empty batch: nothing to launch
  if (!x || !router_w || !ids || !tw) return FLINT_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(router_w, 16) || !aligned(ids, 4) || !aligned(tw, 4))
    return FLINT_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return FLINT_ERR_WORKSPACE;
  const WsLayout L = ws_layout(*shape);
  if (workspace_bytes < L.total) return FLINT_ERR_WORKSPACE;
  MoEArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.router_w = static_cast<const uint16_t*>(router_w);
  a.ids_out = ids;
  a.tw_out = tw;
  a.M = shape->M; a.H = shape->H; a.E = shape->E; a.k = shape->top_k; a.I = shape->I; a.SI = shape->SI;
  a.fault = debug_fault_site();
  a.ws = ws_pointers(workspace, L);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (launch_route(a, false, st, true) != cudaSuccess) return FLINT_ERR_CUDA;
  return FLINT_OK;
}

// Argument checks of the forward entry points (x: the rows the MoE block reads).
static int check_forward(const void* x, const void* router_w, const uint8_t* w13, const uint8_t* w13_sf,
                         const float* w13_gs, const uint8_t* w2, const uint8_t* w2_sf, const float* w2_gs,
                         const void* shared_gu, const void* shared_down, const flint_moe_shape* shape,
                         void* out, int32_t* ids_out, float* tw_out, void* workspace,
                         size_t workspace_bytes) {
  if (!x || !router_w || !w13 || !w13_sf || !w13_gs || !w2 || !w2_sf || !w2_gs || !out)
    return FLINT_ERR_INVALID_ARG;
  if (shape->SI > 0 && (!shared_gu || !shared_down)) return FLINT_ERR_INVALID_ARG;
  const void* p16[] = {x, router_w, w13, w13_sf, w2, w2_sf, out};
  for (const void* p : p16)
    if (!aligned(p, 16)) return FLINT_ERR_INVALID_ARG;
  if (shape->SI > 0 && (!aligned(shared_gu, 16) || !aligned(shared_down, 16)))
    return FLINT_ERR_INVALID_ARG;
  if (!aligned(w13_gs, 4) || !aligned(w2_gs, 4)) return FLINT_ERR_INVALID_ARG;
  if ((ids_out && !aligned(ids_out, 4)) || (tw_out && !aligned(tw_out, 4)))
    return FLINT_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return FLINT_ERR_WORKSPACE;
  if (workspace_bytes < ws_layout(*shape).total) return FLINT_ERR_WORKSPACE;
  return FLINT_OK;
}

// Enqueue the MoE block on rows a.x (arguments checked).
static int enqueue_forward(MoEArgs& a, const flint_moe_shape* shape, cudaStream_t st) {
  int sms = 0;
  if (device_sms(&sms) != cudaSuccess) return FLINT_ERR_CUDA;
  switch (plan(*shape, sms)) {
    case FLINT_PATH_GROUPED:
      if (launch_grouped(a, st) != cudaSuccess) return FLINT_ERR_CUDA;
      return FLINT_OK;
    case FLINT_PATH_SINGLE_LAUNCH:
      if (launch_fused(a, st, sms) != cudaSuccess) return FLINT_ERR_CUDA;
      return FLINT_OK;
    case FLINT_PATH_DECODE:
      if (launch_decode2(a, st) != cudaSuccess) return FLINT_ERR_CUDA;
      return FLINT_OK;
    default:
      if (launch_route(a, true, st, true) != cudaSuccess) return FLINT_ERR_CUDA;
      if (launch_decode_gate_up(a, st, true) != cudaSuccess) return FLINT_ERR_CUDA;
      if (launch_decode_down(a, st, true) != cudaSuccess) return FLINT_ERR_CUDA;
      return FLINT_OK;
  }
}

static MoEArgs make_args(const void* x, const void* router_w, const uint8_t* w13, const uint8_t* w13_sf,
                         const float* w13_gs, const uint8_t* w2, const uint8_t* w2_sf, const float* w2_gs,
                         const void* shared_gu, const void* shared_down, const flint_moe_shape* shape,
                         void* out, int32_t* ids_out, float* tw_out, void* workspace) {
  MoEArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.router_w = static_cast<const uint16_t*>(router_w);
  a.w13 = w13; a.w13_sf = w13_sf; a.w13_gs = w13_gs;
  a.w2 = w2; a.w2_sf = w2_sf; a.w2_gs = w2_gs;
  a.shared_gu = static_cast<const uint16_t*>(shared_gu);
  a.shared_down = static_cast<const uint16_t*>(shared_down);
  a.out = static_cast<uint16_t*>(out);
  a.ids_out = ids_out;
  a.tw_out = tw_out;
  a.M = shape->M; a.H = shape->H; a.E = shape->E; a.k = shape->top_k; a.I = shape->I; a.SI = shape->SI;
  a.fault = debug_fault_site();
  a.ws = ws_pointers(workspace, ws_layout(*shape));
  return a;
}

int flint_moe_forward(const void* x, const void* router_w, const uint8_t* w13, const uint8_t* w13_sf,
                      const float* w13_gs, const uint8_t* w2, const uint8_t* w2_sf,
                      const float* w2_gs, const void* shared_gu, const void* shared_down,
                      const flint_moe_shape* shape, void* out, int32_t* ids_out, float* tw_out,
                      void* workspace, size_t workspace_bytes, flint_stream_t stream) {
  if (!shape_valid(shape)) return FLINT_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return FLINT_ERR_UNSUPPORTED;
  if (shape->M == 0) return FLINT_OK;  // an empty batch: nothing to launch
  const int rc = check_forward(x, router_w, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, shared_gu, shared_down,
                               shape, out, ids_out, tw_out, workspace, workspace_bytes);
  if (rc != FLINT_OK) return rc;
  MoEArgs a = make_args(x, router_w, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, shared_gu, shared_down, shape,
                        out, ids_out, tw_out, workspace);
  return enqueue_forward(a, shape, reinterpret_cast<cudaStream_t>(stream));
}

int flint_moe_forward_add_norm(const void* attn_out, const void* residual, const void* ln_weight, float eps,
                               const void* router_w, const uint8_t* w13, const uint8_t* w13_sf,
                               const float* w13_gs, const uint8_t* w2, const uint8_t* w2_sf,
                               const float* w2_gs, const void* shared_gu, const void* shared_down,
                               const flint_moe_shape* shape, void* out, void* residual_out, void* xn_out,
                               int32_t* ids_out, float* tw_out, void* workspace, size_t workspace_bytes,
                               flint_stream_t stream) {
  if (!shape_valid(shape)) return FLINT_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return FLINT_ERR_UNSUPPORTED;
  if (shape->M == 0) return FLINT_OK;
  if (!attn_out || !residual || !ln_weight || !residual_out) return FLINT_ERR_INVALID_ARG;
  if (!aligned(attn_out, 16) || !aligned(residual, 16) || !aligned(ln_weight, 16) ||
      !aligned(residual_out, 16) || (xn_out && !aligned(xn_out, 16)))
    return FLINT_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || eps > 1.0f) return FLINT_ERR_INVALID_ARG;  // also rejects NaN
  // the MoE block reads the normalised rows: the caller's xn_out, else the
  // workspace's region (checked once the workspace is known to be valid)
  const int rc = check_forward(attn_out, router_w, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, shared_gu,
                               shared_down, shape, out, ids_out, tw_out, workspace, workspace_bytes);
  if (rc != FLINT_OK) return rc;
  MoEArgs a = make_args(nullptr, router_w, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, shared_gu, shared_down,
                        shape, out, ids_out, tw_out, workspace);
  uint16_t* xn = xn_out ? static_cast<uint16_t*>(xn_out) : a.ws.xn;
  a.x = xn;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (launch_add_rms_norm(static_cast<const uint16_t*>(attn_out), static_cast<const uint16_t*>(residual),
                          static_cast<const uint16_t*>(ln_weight), eps, shape->M, shape->H,
                          static_cast<uint16_t*>(residual_out), xn, st) != cudaSuccess)
    return FLINT_ERR_CUDA;
  return enqueue_forward(a, shape, st);
}

int flint_moe_forward_bf16(const void* x, const void* router_w, const void* w13, const void* w2,
                           const void* shared_out, const flint_moe_shape* shape, void* out, int32_t* ids_out,
                           float* tw_out, void* workspace, size_t workspace_bytes, flint_stream_t stream) {
  if (!shape_valid(shape) || shape->SI != 0) return FLINT_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return FLINT_ERR_UNSUPPORTED;
  if (shape->M == 0) return FLINT_OK;
  if (shape->M > kDecodeMaxTokens) return FLINT_ERR_UNSUPPORTED;
  if (!x || !router_w || !w13 || !w2 || !out) return FLINT_ERR_INVALID_ARG;
  const void* p16[] = {x, router_w, w13, w2, out};
  for (const void* p : p16)
    if (!aligned(p, 16)) return FLINT_ERR_INVALID_ARG;
  if (shared_out && !aligned(shared_out, 16)) return FLINT_ERR_INVALID_ARG;
  if ((ids_out && !aligned(ids_out, 4)) || (tw_out && !aligned(tw_out, 4))) return FLINT_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return FLINT_ERR_WORKSPACE;
  if (workspace_bytes < ws_layout(*shape).total) return FLINT_ERR_WORKSPACE;
  MoEArgs a = make_args(x, router_w, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                        shape, out, ids_out, tw_out, workspace);
  if (launch_bf16_experts(a, static_cast<const uint16_t*>(w13), static_cast<const uint16_t*>(w2),
                          static_cast<const uint16_t*>(shared_out),
                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FLINT_ERR_CUDA;
  return FLINT_OK;
}

int flint_moe_forward_nvfp4_shared(const void* x, const void* router_w, const uint8_t* w13,
                                   const uint8_t* w13_sf, const float* w13_gs, const uint8_t* w2,
                                   const uint8_t* w2_sf, const float* w2_gs, const uint8_t* sgu,
                                   const uint8_t* sgu_sf, const float* sgu_gs, const uint8_t* sdown,
                                   const uint8_t* sdown_sf, const float* sdown_gs, const flint_moe_shape* shape,
                                   void* out, int32_t* ids_out, float* tw_out, void* workspace,
                                   size_t workspace_bytes, flint_stream_t stream) {
  if (!shape_valid(shape) || shape->SI < 128) return FLINT_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return FLINT_ERR_UNSUPPORTED;
  if (shape->M == 0) return FLINT_OK;
  if (!sgu || !sgu_sf || !sgu_gs || !sdown || !sdown_sf || !sdown_gs) return FLINT_ERR_INVALID_ARG;
  const void* p16[] = {sgu, sgu_sf, sdown, sdown_sf};
  for (const void* p : p16)
    if (!aligned(p, 16)) return FLINT_ERR_INVALID_ARG;
  if (!aligned(sgu_gs, 4) || !aligned(sdown_gs, 4)) return FLINT_ERR_INVALID_ARG;
  // the routed block: the checks and kernels of flint_moe_forward without a
  // shared expert, on the workspace laid out for the whole shape
  flint_moe_shape routed = *shape;
  routed.SI = 0;
  const int rc = check_forward(x, router_w, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, nullptr, nullptr, &routed,
                               out, ids_out, tw_out, workspace, workspace_bytes);
  if (rc != FLINT_OK) return rc;
  if (workspace_bytes < ws_layout(*shape).total) return FLINT_ERR_WORKSPACE;
  MoEArgs a = make_args(x, router_w, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, nullptr, nullptr, shape, out,
                        ids_out, tw_out, workspace);
  a.SI = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int r = enqueue_forward(a, &routed, st);
  if (r != FLINT_OK) return r;
  if (launch_shared_nvfp4(static_cast<const uint16_t*>(x), sgu, sgu_sf, sgu_gs, sdown, sdown_sf, sdown_gs,
                          shape->M, shape->H, shape->SI, a.ws.sact, a.ws.ys, static_cast<uint16_t*>(out),
                          st) != cudaSuccess)
    return FLINT_ERR_CUDA;
  return FLINT_OK;
}

int flint_moe_plan(const flint_moe_shape* shape) {
  if (!shape_valid(shape)) return FLINT_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return FLINT_ERR_UNSUPPORTED;
  if (shape->M == 0) return FLINT_PATH_NONE;
  int sms = 0;
  if (device_sms(&sms) != cudaSuccess) return FLINT_ERR_CUDA;
  return plan(*shape, sms);
}

int flint_moe_status(void* workspace, flint_stream_t stream) {
  if (!workspace) return FLINT_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FLINT_ERR_CUDA;
  int status = 0;
  if (cudaMemcpy(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FLINT_ERR_CUDA;
  if (status != 0) {
    if (cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return FLINT_ERR_CUDA;
    return status;
  }
  return FLINT_OK;
}

int flint_moe_prefer_path(int path) {
  if (path != FLINT_PATH_NONE && path != FLINT_PATH_SINGLE_LAUNCH) return FLINT_ERR_INVALID_ARG;
  g_prefer.store(path, std::memory_order_relaxed);
  return FLINT_OK;
}

int flint_moe_record_spans(unsigned long long* spans) {
  cudaError_t (*const set[])(unsigned long long*) = {span_buffer_set_decode2, span_buffer_set_decode,
                                                     span_buffer_set_fused, span_buffer_set_grouped,
                                                     span_buffer_set_route, span_buffer_set_add_norm,
                                                     span_buffer_set_bf16_experts,
                                                     span_buffer_set_shared_nvfp4, span_buffer_set_qkv};
  for (auto f : set)
    if (f(spans) != cudaSuccess) return FLINT_ERR_CUDA;
  return FLINT_OK;
}

// ---------------------------------------------------------- fused qkv --
// Workspace: status word (offset 0, read by flint_moe_status), xn [M, H],
// qkv [M, (nq + 2 nkv) * 128], each region 256-byte aligned.
static size_t qkv_ws(int M, int H, int nq, int nkv, size_t* xn_off, size_t* qkv_off) {
  auto al = [](size_t v) { return (v + 255) / 256 * 256; };
  const size_t xo = 256, qo = xo + al((size_t)M * H * 2);
  if (xn_off) *xn_off = xo;
  if (qkv_off) *qkv_off = qo;
  return qo + al((size_t)M * (nq + 2 * nkv) * 128 * 2);
}

size_t flint_qkv_workspace_bytes(int M, int H, int num_q_heads, int num_kv_heads) {
  if (M < 0 || H <= 0 || H % 128 != 0 || num_q_heads < 1 || num_kv_heads < 0) return 0;
  return qkv_ws(M, H, num_q_heads, num_kv_heads, nullptr, nullptr);
}

int flint_qkv_fused(const void* x, const void* residual, const void* norm_weight, float eps,
                    const void* weight, const uint8_t* weight_scale, const float* global_scale,
                    const void* q_norm_weight, const void* k_norm_weight, float qk_eps,
                    const float* cos_sin_cache, long long max_pos, const long long* positions,
                    void* k_cache, void* v_cache, long long stride_block, long long stride_slot,
                    long long stride_head, int block_size, long long num_blocks,
                    const long long* slot_mapping, int num_slots, int M, int H, int num_q_heads,
                    int num_kv_heads, void* q_out, void* residual_out, void* workspace, size_t ws_bytes,
                    flint_stream_t stream) {
  if (M < 0 || H <= 0 || H % 64 != 0 || num_q_heads < 1 || num_kv_heads < 0 || num_slots < 0)
    return FLINT_ERR_INVALID_ARG;
  if (H % 128 != 0) return FLINT_ERR_UNSUPPORTED;
  if (M == 0) return FLINT_OK;
  if (!x || !norm_weight || !weight || !q_norm_weight || !q_out) return FLINT_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(norm_weight, 16) || !aligned(weight, 16) || !aligned(q_out, 16) ||
      !aligned(q_norm_weight, 2))
    return FLINT_ERR_INVALID_ARG;
  if (residual && (!aligned(residual, 16) || !residual_out || !aligned(residual_out, 16)))
    return FLINT_ERR_INVALID_ARG;
  if (weight_scale && (!global_scale || !aligned(global_scale, 4))) return FLINT_ERR_INVALID_ARG;
  if (cos_sin_cache && (!positions || max_pos < 1 || !aligned(cos_sin_cache, 4) || !aligned(positions, 8)))
    return FLINT_ERR_INVALID_ARG;
  if (num_kv_heads > 0 && (!k_norm_weight || !aligned(k_norm_weight, 2))) return FLINT_ERR_INVALID_ARG;
  const bool writes = num_kv_heads > 0 && num_slots > 0;
  if (writes && (!k_cache || !v_cache || !slot_mapping || !aligned(k_cache, 2) || !aligned(v_cache, 2) ||
                 !aligned(slot_mapping, 8) || block_size < 1 || num_blocks < 0 || stride_block < 0 ||
                 stride_slot < 0 || stride_head < 0))
    return FLINT_ERR_INVALID_ARG;
  size_t xo = 0, qo = 0;
  const size_t need = qkv_ws(M, H, num_q_heads, num_kv_heads, &xo, &qo);
  if (!workspace || !aligned(workspace, 256) || ws_bytes < need) return FLINT_ERR_WORKSPACE;
  uint8_t* wb = static_cast<uint8_t*>(workspace);
  QkvArgs a = {};
  a.M = M; a.H = H; a.nq = num_q_heads; a.nkv = num_kv_heads;
  a.q_norm_w = static_cast<const uint16_t*>(q_norm_weight);
  a.k_norm_w = static_cast<const uint16_t*>(k_norm_weight);
  a.qk_eps = qk_eps;
  a.cos_sin = cos_sin_cache;
  a.max_pos = max_pos;
  a.positions = positions;
  a.slot_mapping = writes ? slot_mapping : nullptr;
  a.n_slots = writes ? num_slots : 0;
  a.k_cache = static_cast<uint16_t*>(k_cache);
  a.v_cache = static_cast<uint16_t*>(v_cache);
  a.s_block = stride_block; a.s_slot = stride_slot; a.s_head = stride_head;
  a.block_size = block_size > 0 ? block_size : 1;
  a.num_blocks = num_blocks;
  a.q_out = static_cast<uint16_t*>(q_out);
  a.xn = reinterpret_cast<uint16_t*>(wb + xo);
  a.qkv = reinterpret_cast<uint16_t*>(wb + qo);
  a.status = reinterpret_cast<int*>(wb);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t err =
      launch_qkv_fused(a, static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(residual),
                       static_cast<const uint16_t*>(norm_weight), eps, weight, weight_scale, global_scale,
                       residual ? static_cast<uint16_t*>(residual_out) : nullptr, st);
  return err == cudaSuccess ? FLINT_OK : FLINT_ERR_CUDA;
}

int flint_moe_debug_fault(int site) {
  if (site != FLINT_FAULT_NONE && site != FLINT_FAULT_DOWN_HANDOVER) return FLINT_ERR_INVALID_ARG;
  g_fault_site.store(site, std::memory_order_relaxed);
  return FLINT_OK;
}

const char* flint_moe_strerror(int code) {
  switch (code) {
    case FLINT_OK: return "ok";
    case FLINT_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, or bad shape)";
    case FLINT_ERR_UNSUPPORTED: return "shape not supported by the kernels";
    case FLINT_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case FLINT_ERR_CUDA: return "CUDA runtime or launch error";
    case FLINT_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    case FLINT_ERR_SCRATCH: return "shape needs more than the library's fixed static scratch";
    default: return "unknown error";
  }
}

}  // extern "C"
