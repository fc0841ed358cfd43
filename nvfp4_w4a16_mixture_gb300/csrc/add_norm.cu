// Add-RMSNorm prologue of the decode MoE block.
//
// Page "vllm.models.flint.ops.moe": flint_moe_ll computes
// residual' = attn_out + residual and x = rms_norm(residual') as
// norm.fused_add_rms_norm (_add_rms_norm on that page: both outputs from the
// unrounded fp32 sum s = a + r, inv = rsqrt(mean(s^2) + eps),
// xn = bf16(s * inv * w)), then runs the MoE block on x.
//
// One warp per token.  The sum of squares is taken in double (every fp32
// square is exact there, and the sum of at most a few thousand of them is
// within a unit of the 50th bit of the exact sum), rounded once to fp32;
// inv is 1 / sqrt(v) in double rounded once to fp32, which is the correctly
// rounded reciprocal square root but for inputs within 2^-29 of an fp32
// rounding boundary.
#include "common.cuh"
#include "internal.h"

namespace flint {
namespace {

constexpr int kNormWarps = 8;

__global__ void __launch_bounds__(kNormWarps * 32) add_rms_norm_kernel(
    const uint16_t* __restrict__ a, const uint16_t* __restrict__ r, const uint16_t* __restrict__ w,
    float eps, int M, int H, uint16_t* __restrict__ res_out, uint16_t* __restrict__ xn) {
  SpanGuard<kSpanAddNorm> span_guard;
  pdl_wait();  // the inputs belong to the stream's earlier work
  pdl_launch_dependents();
  const int t = blockIdx.x * kNormWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= M) return;
  const uint16_t* at = a + (size_t)t * H;
  const uint16_t* rt = r + (size_t)t * H;
  double sq = 0.0;
  for (int h = 8 * lane; h < H; h += 256) {
    const uint4 av = ldg_nc_v4(at + h), rv = ldg_nc_v4(rt + h);
    const uint32_t aw[4] = {av.x, av.y, av.z, av.w}, rw[4] = {rv.x, rv.y, rv.z, rv.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float s0 = __fadd_rn(__uint_as_float(aw[q] << 16), __uint_as_float(rw[q] << 16));
      const float s1 = __fadd_rn(__uint_as_float(aw[q] & 0xFFFF0000u), __uint_as_float(rw[q] & 0xFFFF0000u));
      o[q] = f32_to_bf16_bits(s0) | (f32_to_bf16_bits(s1) << 16);
      sq = fma((double)s0, (double)s0, sq);
      sq = fma((double)s1, (double)s1, sq);
    }
    *reinterpret_cast<uint4*>(res_out + (size_t)t * H + h) = make_uint4(o[0], o[1], o[2], o[3]);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
  const float v = __fadd_rn(__fdiv_rn((float)sq, (float)H), eps);
  const float inv = (float)(1.0 / sqrt((double)v));
  for (int h = 8 * lane; h < H; h += 256) {
    const uint4 av = ldg_nc_v4(at + h), rv = ldg_nc_v4(rt + h), wv = ldg_nc_v4(w + h);
    const uint32_t aw[4] = {av.x, av.y, av.z, av.w}, rw[4] = {rv.x, rv.y, rv.z, rv.w};
    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float s0 = __fadd_rn(__uint_as_float(aw[q] << 16), __uint_as_float(rw[q] << 16));
      const float s1 = __fadd_rn(__uint_as_float(aw[q] & 0xFFFF0000u), __uint_as_float(rw[q] & 0xFFFF0000u));
      const float x0 = __fmul_rn(__fmul_rn(s0, inv), __uint_as_float(ww[q] << 16));
      const float x1 = __fmul_rn(__fmul_rn(s1, inv), __uint_as_float(ww[q] & 0xFFFF0000u));
      o[q] = f32_to_bf16_bits(x0) | (f32_to_bf16_bits(x1) << 16);
    }
    *reinterpret_cast<uint4*>(xn + (size_t)t * H + h) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_add_rms_norm(const uint16_t* a, const uint16_t* r, const uint16_t* w, float eps,
                                int M, int H, uint16_t* res_out, uint16_t* xn, cudaStream_t st) {
  void* args[] = {&a, &r, &w, &eps, &M, &H, &res_out, &xn};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((M + kNormWarps - 1) / kNormWarps));
  cfg.blockDim = dim3(kNormWarps * 32);
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
