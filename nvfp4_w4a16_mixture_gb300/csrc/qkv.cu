// Fused decode qkv: input RMSNorm, the qkv GEMV, per-head q/k RMSNorm, NeoX
// RoPE and the paged KV-cache write.
//
// Page "vllm.models.flint.ops.qkv_fused": flint_qkv_fused runs
// fused_add_rms_norm (rms_norm for the first layer) writing xn and the new
// residual, then the qkv GEMV over xn (NVFP4 codes with e4m3 block scales
// and an fp32 global scale, or BF16 weights), whose rows are the q heads,
// then the k heads, then the v heads (128 each); q and k heads get an
// RMSNorm over their 128 values with the per-head weights and NeoX RoPE from
// an fp32 cos | sin table at the token's position, fp32 math; k and v go to
// the paged caches at slot_mapping[t] (negative slots, and tokens past the
// mapping, are not written), q to the output.
//
// Three launches chained with programmatic dependent launch: the input norm
// (add_norm.cu), the GEMV (CTA: 16 weight rows x 64 tokens, its 8 warps over
// the token tiles and, for few tokens, over K; every sum exact as in the
// decode kernels, exact.cuh), and the head kernel (one warp per token and
// head).  The GEMV rounds each value to BF16 (times the global scale on the
// fp32 sum for NVFP4 weights); the head kernel sums the squares of a head's
// 128 BF16 values in double (exact), rounds the sum once, takes inv = 1 /
// sqrt in double rounded once, n = (q * inv) * w in fp32, then
// o[d] = n[d] c - n[d + 64] s, o[d + 64] = n[d + 64] c + n[d] s (each
// product and sum one fp32 rounding) and rounds o to BF16.
#include "common.cuh"
#include "exact.cuh"
#include "frag.cuh"
#include "internal.h"

namespace flint {
namespace {

constexpr int kQkvWarps = 8;  // 2 CTAs per SM: 320 CTAs of the N = 5120 GEMV in one wave
constexpr int kHead = 128;
constexpr int kHeadWarps = 4;

FLINT_DEV void load_act(uint4 (&xb)[4], const uint16_t* p) {
#pragma unroll
  for (int q = 0; q < 4; ++q) xb[q] = p ? ldg_cg_v4(p + 8 * q) : make_uint4(0, 0, 0, 0);
}

// out[t, n] for n in 16 blockIdx.x .. + 15, t in 64 blockIdx.y .. + 63:
// bf16(fp32(exact dot(act[t], W[n])) * gs) (NVFP4: codes [N, K/2], scales
// [N, K/16]) or bf16(fp32(exact dot)) (BF16: [N, K]).
template <bool NVFP4>
__global__ void __launch_bounds__(kQkvWarps * 32) qkv_gemv_kernel(
    const uint16_t* __restrict__ act, const void* __restrict__ w, const uint8_t* __restrict__ sf,
    const float* __restrict__ gs_p, int M, int N, int K, uint16_t* __restrict__ out) {
  SpanGuard<kSpanQkvGemv> span_guard;
  pdl_wait();  // xn is the previous kernel's output
  pdl_launch_dependents();
  __shared__ float4 red[kQkvWarps * 64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int ntiles = (min(64, M - 64 * (int)blockIdx.y) + 7) / 8;
  const int kw = max(1, kQkvWarps / ntiles), tile = warp / kw, part = warp % kw;
  const bool active = tile < ntiles;
  const int t0 = 64 * blockIdx.y + 8 * tile;
  const int n0 = 16 * blockIdx.x;
  const int tok = t0 + g;
  const uint16_t* arow = active && tok < M ? act + (size_t)tok * K : nullptr;
  float S[4] = {0.0f, 0.0f, 0.0f, 0.0f}, C[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int s = part; active && s < K / kSliceK; s += kw) {
    uint4 xb[4];
    load_act(xb, arow ? arow + s * kSliceK + 32 * t : nullptr);
    if constexpr (NVFP4) {
      const uint8_t* codes = static_cast<const uint8_t*>(w);
      const uint8_t* ca = codes + (size_t)(n0 + g) * (K / 2);
      const uint8_t* cb = codes + (size_t)(n0 + 8 + g) * (K / 2);
      const uint8_t* sa = sf + (size_t)(n0 + g) * (K / 16);
      const uint8_t* sb = sf + (size_t)(n0 + 8 + g) * (K / 16);
      slice_nvfp4_exact(S, C, ca + s * (kSliceK / 2) + 16 * t, cb + s * (kSliceK / 2) + 16 * t,
                        *reinterpret_cast<const uint16_t*>(sa + s * (kSliceK / 16) + 2 * t),
                        *reinterpret_cast<const uint16_t*>(sb + s * (kSliceK / 16) + 2 * t), xb);
    } else {
      const uint16_t* wb = static_cast<const uint16_t*>(w);
      slice_bf16_exact(S, C, wb + (size_t)(n0 + g) * K + s * kSliceK + 32 * t,
                       wb + (size_t)(n0 + 8 + g) * K + s * kSliceK + 32 * t, xb);
    }
  }
  if (kw > 1) {
    store_pair(red, warp, lane, S, C);
    __syncthreads();
    if (!active || part != 0) return;
    add_pairs(S, C, red, warp, kw, lane);
  } else if (!active) {
    return;
  }
  // the NVFP4 slices summed the weights times 2^-7: scale back exactly, then
  // the global scale on the fp32 sum
  const float gs = NVFP4 ? *gs_p : 1.0f;
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int tt = t0 + 2 * t + cc;
    if (tt < M) {
      float v0 = __fadd_rn(S[cc], C[cc]), v1 = __fadd_rn(S[2 + cc], C[2 + cc]);
      if (NVFP4) {
        v0 = __fmul_rn(v0 * 128.0f, gs);
        v1 = __fmul_rn(v1 * 128.0f, gs);
      }
      out[(size_t)tt * N + n0 + g] = (uint16_t)f32_to_bf16_bits(v0);
      out[(size_t)tt * N + n0 + 8 + g] = (uint16_t)f32_to_bf16_bits(v1);
    }
  }
}

// Records an argument error found on the device (the first one wins).
FLINT_DEV void qkv_error(int* status) { atomicCAS(status, 0, FLINT_ERR_INVALID_ARG); }

// One warp per (token, head): lane l holds dims l, l + 32, l + 64, l + 96,
// so each of its two NeoX pairs (d, d + 64) sits in one lane.
__global__ void __launch_bounds__(kHeadWarps * 32) qkv_heads_kernel(QkvArgs a) {
  SpanGuard<kSpanQkvHeads> span_guard;
  pdl_wait();  // qkv is the previous kernel's output
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nh = a.nq + 2 * a.nkv;
  const int gid = blockIdx.x * kHeadWarps + warp;
  if (gid >= a.M * nh) return;
  const int t = gid / nh, hh = gid % nh;
  const int N = nh * kHead;
  const uint16_t* row = a.qkv + (size_t)t * N + (size_t)hh * kHead;
  uint32_t vb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) vb[i] = row[lane + 32 * i];
  // the token's cache row (slot < 0 or past the mapping: not written)
  long long slot = t < a.n_slots ? a.slot_mapping[t] : -1;
  if (slot >= (long long)a.num_blocks * a.block_size) {
    if (lane == 0) qkv_error(a.status);
    slot = -1;
  }
  uint16_t* kv_row = nullptr;
  if (slot >= 0 && hh >= a.nq) {
    const long long blk = slot / a.block_size, off = slot % a.block_size;
    const int kvh = hh < a.nq + a.nkv ? hh - a.nq : hh - a.nq - a.nkv;
    kv_row = (hh < a.nq + a.nkv ? a.k_cache : a.v_cache) + blk * a.s_block + off * a.s_slot +
             (long long)kvh * a.s_head;
  }
  if (hh >= a.nq + a.nkv) {  // v head: the qkv values as they are
    if (kv_row) {
#pragma unroll
      for (int i = 0; i < 4; ++i) kv_row[lane + 32 * i] = (uint16_t)vb[i];
    }
    return;
  }
  float v[4];
  double sq = 0.0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = bf16_bits_to_f32(vb[i]);
    sq = fma((double)v[i], (double)v[i], sq);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  const float var = __fadd_rn(__fdiv_rn((float)sq, (float)kHead), a.qk_eps);
  const float inv = (float)(1.0 / sqrt((double)var));
  const uint16_t* nw = hh < a.nq ? a.q_norm_w : a.k_norm_w;
  float n[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) n[i] = __fmul_rn(__fmul_rn(v[i], inv), bf16_bits_to_f32(nw[lane + 32 * i]));
  float o[4] = {n[0], n[1], n[2], n[3]};
  if (a.cos_sin) {
    const long long pos = a.positions[t];
    if (pos < 0 || pos >= a.max_pos) {
      if (lane == 0) qkv_error(a.status);
    } else {
      const float* cs = a.cos_sin + pos * kHead;
#pragma unroll
      for (int i = 0; i < 2; ++i) {  // pairs (l + 32 i, l + 32 i + 64)
        const float c = cs[lane + 32 * i], s = cs[kHead / 2 + lane + 32 * i];
        o[i] = __fsub_rn(__fmul_rn(n[i], c), __fmul_rn(n[i + 2], s));
        o[i + 2] = __fadd_rn(__fmul_rn(n[i + 2], c), __fmul_rn(n[i], s));
      }
    }
  }
  uint16_t* dst = hh < a.nq ? a.q_out + (size_t)t * a.nq * kHead + (size_t)hh * kHead : kv_row;
  if (dst) {
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = (uint16_t)f32_to_bf16_bits(o[i]);
  }
}

cudaError_t launch_pdl_qkv(const void* fn, dim3 grid, dim3 block, void** args, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

cudaError_t launch_qkv_fused(const QkvArgs& a, const uint16_t* x, const uint16_t* residual,
                             const uint16_t* norm_w, float eps, const void* w, const uint8_t* w_sf,
                             const float* gs, uint16_t* res_out, cudaStream_t st) {
  cudaError_t err = launch_add_rms_norm(x, residual, norm_w, eps, a.M, a.H, res_out, a.xn, st);
  if (err != cudaSuccess) return err;
  const int N = (a.nq + 2 * a.nkv) * kHead;
  const uint16_t* act = a.xn;
  int M = a.M, H = a.H;
  uint16_t* out = a.qkv;
  void* g_args[] = {(void*)&act, (void*)&w, (void*)&w_sf, (void*)&gs, &M, (void*)&N, &H, &out};
  const void* fn = w_sf ? (const void*)qkv_gemv_kernel<true> : (const void*)qkv_gemv_kernel<false>;
  err = launch_pdl_qkv(fn, dim3((unsigned)(N / 16), (unsigned)((M + 63) / 64)), dim3(kQkvWarps * 32), g_args, st);
  if (err != cudaSuccess) return err;
  QkvArgs aa = a;
  void* h_args[] = {&aa};
  const long long warps = (long long)a.M * (a.nq + 2 * a.nkv);
  return launch_pdl_qkv((const void*)qkv_heads_kernel, dim3((unsigned)((warps + kHeadWarps - 1) / kHeadWarps)),
                        dim3(kHeadWarps * 32), h_args, st);
}

FLINT_SPAN_SETTER(qkv)

}  // namespace flint
