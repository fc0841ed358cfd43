// Add-RMSNorm prologue of the decode MoE block.
//
// Page "vllm.models.flint.ops.moe": flint_moe_ll computes
// residual' = attn_out + residual and x = rms_norm(residual') as
// norm.fused_add_rms_norm (_add_rms_norm on that page: both outputs from the
// unrounded fp32 sum s = a + r, inv = rsqrt(mean(s^2) + eps),
// xn = bf16(s * inv * w)), then runs the MoE block on x.
//
// Without a residual (r == nullptr) it is the plain RMSNorm of a, and
// res_out (then optional) is not written.
//
// One CTA of 8 warps per token, each thread a few 8-element vectors of the
// row, kept in registers between the two passes (rows up to 4096 wide; the
// rest of a wider row is read again).  The sum of squares is taken in double
// (every fp32 square is exact there, and the sum of at most a few thousand of
// them is within a unit of the 50th bit of the exact sum), rounded once to
// fp32; inv is 1 / sqrt(v) in double rounded once to fp32, which is the
// correctly rounded reciprocal square root but for inputs within 2^-29 of an
// fp32 rounding boundary.  The next kernel (the router) is released at once:
// it loads its weights and then waits for this grid.
#include "common.cuh"
#include "internal.h"

namespace flint {
namespace {

constexpr int kNormThreads = 256;
constexpr int kNormCache = 2;  // row vectors kept in registers per thread

// s = a + r in fp32 (r == nullptr: s = a, no addition)
FLINT_DEV void add_vec(const uint16_t* ap, const uint16_t* rp, float (&s)[8]) {
  const uint4 av = ldg_nc_v4(ap);
  const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
  if (!rp) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      s[2 * q] = __uint_as_float(aw[q] << 16);
      s[2 * q + 1] = __uint_as_float(aw[q] & 0xFFFF0000u);
    }
    return;
  }
  const uint4 rv = ldg_nc_v4(rp);
  const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    s[2 * q] = __fadd_rn(__uint_as_float(aw[q] << 16), __uint_as_float(rw[q] << 16));
    s[2 * q + 1] = __fadd_rn(__uint_as_float(aw[q] & 0xFFFF0000u), __uint_as_float(rw[q] & 0xFFFF0000u));
  }
}

__global__ void __launch_bounds__(kNormThreads) add_rms_norm_kernel(
    const uint16_t* __restrict__ a, const uint16_t* __restrict__ r, const uint16_t* __restrict__ w,
    float eps, int M, int H, uint16_t* __restrict__ res_out, uint16_t* __restrict__ xn) {
  SpanGuard<kSpanAddNorm> span_guard;
  pdl_launch_dependents();  // the router waits for this grid before it reads xn
  pdl_wait();               // the inputs belong to the stream's earlier work
  __shared__ double part[kNormThreads / 32];
  __shared__ float s_inv;
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint16_t* at = a + (size_t)t * H;
  const uint16_t* rt = r ? r + (size_t)t * H : nullptr;  // no residual: plain RMSNorm
  const int nv = H / 8;  // 8-element vectors of the row
  float cache[kNormCache][8];
  double sq0 = 0.0, sq1 = 0.0;
  for (int v = tid, i = 0; v < nv; v += kNormThreads, ++i) {
    float sv[8];
    add_vec(at + 8 * v, rt ? rt + 8 * v : nullptr, sv);
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      o[q] = f32_to_bf16_bits(sv[2 * q]) | (f32_to_bf16_bits(sv[2 * q + 1]) << 16);
      sq0 = fma((double)sv[2 * q], (double)sv[2 * q], sq0);
      sq1 = fma((double)sv[2 * q + 1], (double)sv[2 * q + 1], sq1);
    }
    if (res_out)
      *reinterpret_cast<uint4*>(res_out + (size_t)t * H + 8 * v) = make_uint4(o[0], o[1], o[2], o[3]);
#pragma unroll
    for (int c = 0; c < kNormCache; ++c)
      if (c == i)
#pragma unroll
        for (int j = 0; j < 8; ++j) cache[c][j] = sv[j];
  }
  double sq = sq0 + sq1;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
  if (lane == 0) part[warp] = sq;
  __syncthreads();
  if (tid == 0) {
    double tot = 0.0;
    for (int i = 0; i < kNormThreads / 32; ++i) tot += part[i];
    const float v = __fadd_rn(__fdiv_rn((float)tot, (float)H), eps);
    s_inv = (float)(1.0 / sqrt((double)v));
  }
  __syncthreads();
  const float inv = s_inv;
  for (int v = tid, i = 0; v < nv; v += kNormThreads, ++i) {
    float sv[8];
    if (i < kNormCache) {
#pragma unroll
      for (int c = 0; c < kNormCache; ++c)
        if (c == i)
#pragma unroll
          for (int j = 0; j < 8; ++j) sv[j] = cache[c][j];
    } else {
      add_vec(at + 8 * v, rt ? rt + 8 * v : nullptr, sv);
    }
    const uint4 wv = ldg_nc_v4(w + 8 * v);
    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float x0 = __fmul_rn(__fmul_rn(sv[2 * q], inv), __uint_as_float(ww[q] << 16));
      const float x1 = __fmul_rn(__fmul_rn(sv[2 * q + 1], inv), __uint_as_float(ww[q] & 0xFFFF0000u));
      o[q] = f32_to_bf16_bits(x0) | (f32_to_bf16_bits(x1) << 16);
    }
    *reinterpret_cast<uint4*>(xn + (size_t)t * H + 8 * v) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_add_rms_norm(const uint16_t* a, const uint16_t* r, const uint16_t* w, float eps,
                                int M, int H, uint16_t* res_out, uint16_t* xn, cudaStream_t st) {
  void* args[] = {&a, &r, &w, &eps, &M, &H, &res_out, &xn};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M);
  cfg.blockDim = dim3(kNormThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, (const void*)add_rms_norm_kernel, args);
}

FLINT_SPAN_SETTER(add_norm)

}  // namespace flint
