// Router GEMV + top-k + expert grouping.
//
// Router logits, top-k, sigmoid renormalisation: vLLM page
// "vllm.models.flint.ops.moe", _router_kernel / _topk_row docstrings (BF16
// logits, ties to the lowest expert index, s / (sum + 1e-20) rounded to
// BF16).  Expert grouping (histogram, exclusive scan, stable scatter of the
// (token, slot) pairs by expert) is the token permutation the grouped path of
// flint_moe consumes ("perm" of _combine_kernel); the decode path uses the
// same grouping to stream each routed expert's weights once per call.
#include "common.cuh"
#include "internal.h"

namespace flint {

constexpr int kRouteWarps = 4;  // one expert per warp

// ----------------------------------------------------------------------------
// Expert grouping for small M, run by one CTA of >= 128 threads.
// sorted_pairs lists the pairs p = t * k + j of each expert in ascending p
// (experts ascending); rowof[p] is the inverse.
__device__ void build_groups_small(const MoEArgs& a, const int* ids, int* rowof) {
  __shared__ uint8_t s_pos[kDecodeMaxTokens][kMaxE];  // slot j of expert e in token t, 0xFF = none
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_uoff[kMaxE + 1];
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int M = a.M, E = a.E, k = a.k, np = M * k;
  for (int i = tid; i < kDecodeMaxTokens * kMaxE / 4; i += nthr)
    reinterpret_cast<uint32_t*>(&s_pos[0][0])[i] = 0xFFFFFFFFu;
  for (int e = tid; e < kMaxE; e += nthr) s_cnt[e] = 0;
  __syncthreads();
  for (int p = tid; p < np; p += nthr) {
    int e = ldg_cg_i32(ids + p);
    s_pos[p / k][e] = (uint8_t)(p % k);
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  if (tid < 32) {  // exclusive scans of counts and of "routed" flags, one warp
    int run = 0, urun = 0;
    for (int base = 0; base < E; base += 32) {
      int e = base + tid;
      int c = e < E ? s_cnt[e] : 0;
      int u = c > 0 ? 1 : 0;
      int ic = c, iu = u;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int vc = __shfl_up_sync(0xffffffffu, ic, o);
        int vu = __shfl_up_sync(0xffffffffu, iu, o);
        if (tid >= o) { ic += vc; iu += vu; }
      }
      if (e < E) { s_off[e] = run + ic - c; s_uoff[e] = urun + iu - u; }
      run += __shfl_sync(0xffffffffu, ic, 31);
      urun += __shfl_sync(0xffffffffu, iu, 31);
    }
    if (tid == 0) { s_off[E] = run; s_uoff[E] = urun; }
  }
  __syncthreads();
  for (int e = tid; e < E; e += nthr) {
    a.ws.e_cnt[e] = s_cnt[e];
    a.ws.e_off[e] = s_off[e];
    if (s_cnt[e] > 0) a.ws.uniq[1 + s_uoff[e]] = e;
    int c = s_off[e];
    for (int t = 0; t < M; ++t) {
      int j = s_pos[t][e];
      if (j != 0xFF) {
        int p = t * k + j;
        a.ws.sorted_pairs[c] = p;
        rowof[p] = c;
        ++c;
      }
    }
  }
  if (tid == 0) { a.ws.e_off[E] = s_off[E]; a.ws.uniq[0] = s_uoff[E]; }
}

// ----------------------------------------------------------------------------
// Router logits: grid (ceil(E / 4), ceil(M / kRouteTokens)), 4 warps, warp w
// computes expert blockIdx.x * 4 + w for the CTA's tokens.  Lane l owns the
// elements h with (h / 8) mod 32 == l: per 256-wide chunk c one 16-byte
// vector at h = 256 c + 8 l; its fp32 partial sum runs over (c, i) ascending
// with fmaf (each bf16 x bf16 product is exact in fp32, so fmaf is one
// rounded add).  The 32 partials are combined by the xor butterfly with
// offsets 16, 8, 4, 2, 1 and lane 0's value is rounded to BF16.  This fixed
// order is what makes the ids reproducible bit for bit.
//
// The last CTA (atomic counter) of each token block then runs top-k for the
// block's tokens; with build_meta, the last token block's finisher builds the
// expert grouping (M <= kDecodeMaxTokens).
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(MoEArgs a, int build_meta,
                                                                 int* rowof) {
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouteWarps + warp;
  const int tb = blockIdx.y;
  const int H = a.H, E = a.E, k = a.k;
  const int t0 = tb * kRouteTokens;
  const int nt = min(kRouteTokens, a.M - t0);
  const int nchunk = (H + 255) / 256;
  const bool active = e < E;
  const uint16_t* wrow = a.router_w + (size_t)(active ? e : 0) * H;

  // router weights do not depend on earlier grids: fetch before the wait
  uint4 wreg[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    int h = 256 * c + 8 * lane;
    wreg[c] = (active && c < nchunk && h < H && H <= 2048) ? ldg_nc_v4(wrow + h) : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();

  if (active) {
    for (int tt = 0; tt < nt; ++tt) {
      const uint16_t* xrow = a.x + (size_t)(t0 + tt) * H;
      float acc = 0.0f;
      for (int c = 0; c < nchunk; ++c) {
        int h = 256 * c + 8 * lane;
        if (h < H) {
          uint4 xv = ldg_cg_v4(xrow + h);
          uint4 wv;
          if (H <= 2048) {
            wv = wreg[0];
#pragma unroll
            for (int cc = 1; cc < 8; ++cc)
              if (cc == c) wv = wreg[cc];
          } else {
            wv = ldg_nc_v4(wrow + h);
          }
          const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
          const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc = fmaf(__uint_as_float(xs[q] << 16), __uint_as_float(ws[q] << 16), acc);
            acc = fmaf(__uint_as_float(xs[q] & 0xFFFF0000u), __uint_as_float(ws[q] & 0xFFFF0000u), acc);
          }
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) acc = acc + __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) a.ws.logits[(size_t)(t0 + tt) * E + e] = (uint16_t)f32_to_bf16_bits(acc);
    }
  }

  // ---- last CTA of this token block: top-k for its tokens
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    int old = atomicAdd(&a.ws.tok_cnt[tb], 1);
    s_last = (old == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) a.ws.tok_cnt[tb] = 0;  // ready for the next launch

  for (int tt = warp; tt < nt; tt += kRouteWarps) {
    const int t = t0 + tt;
    // key = (order-preserving bf16 bits << 8) | (E - 1 - e): max key = largest
    // logit, lowest expert index among equal bit patterns
    int key[kMaxE / 32];
#pragma unroll
    for (int q = 0; q < kMaxE / 32; ++q) {
      int ee = q * 32 + lane;
      key[q] = -1;
      if (ee < E) {
        uint32_t b = ldg_cg_u16(a.ws.logits + (size_t)t * E + ee);
        key[q] = (int)((ordered_bf16(b) << 8) | (uint32_t)(E - 1 - ee));
      }
    }
    float sum = 0.0f, my_s = 0.0f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
      int lm = key[0];
#pragma unroll
      for (int q = 1; q < kMaxE / 32; ++q) lm = max(lm, key[q]);
      const int best = __reduce_max_sync(0xffffffffu, lm);
#pragma unroll
      for (int q = 0; q < kMaxE / 32; ++q)
        if (key[q] == best) key[q] = -1;
      const uint32_t o = (uint32_t)best >> 8;
      const uint32_t b16 = (o & 0x8000u) ? (o ^ 0x8000u) : (o ^ 0xFFFFu);
      const float logit = bf16_bits_to_f32(b16);
      const float s = __fdiv_rn(1.0f, 1.0f + expf(-logit));
      sum = sum + s;  // rank order
      if (lane == j) { my_s = s; my_e = E - 1 - (best & 0xFF); }
    }
    if (lane < k) {
      const float w = round_bf16(__fdiv_rn(my_s, sum + 1e-20f));
      a.ws.ids[t * k + lane] = my_e;
      a.ws.tw[t * k + lane] = w;
      if (a.ids_out) a.ids_out[t * k + lane] = my_e;
      if (a.tw_out) a.tw_out[t * k + lane] = w;
    }
  }
  if (!build_meta) return;

  // ---- last token block to finish: expert grouping for all tokens
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    int old = atomicAdd(&a.ws.glob_cnt[0], 1);
    s_last = (old == (int)gridDim.y - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) a.ws.glob_cnt[0] = 0;
  build_groups_small(a, a.ws.ids, rowof);
}

// ----------------------------------------------------------------------------
// Expert grouping for any M, three kernels over chunks of kGroupChunk pairs:
//   group_count: per-chunk expert histogram        -> ccnt[chunk][E]
//   group_scan:  expert offsets, per-chunk offsets -> e_cnt, e_off, uniq, coff
//   group_scatter: stable scatter inside each chunk -> sorted_pairs, rowof
constexpr int kGroupChunk = 1024;
constexpr int kGroupThreads = 256;

__global__ void __launch_bounds__(kGroupThreads) group_count_kernel(MoEArgs a, int* ccnt) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int s_cnt[kMaxE];
  const int E = a.E, np = a.M * a.k;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kGroupChunk;
  for (int i = threadIdx.x; i < kGroupChunk; i += blockDim.x) {
    int p = p0 + i;
    if (p < np) atomicAdd(&s_cnt[ldg_cg_i32(a.ws.ids + p)], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) ccnt[(size_t)blockIdx.x * E + e] = s_cnt[e];
}

// One CTA: thread e walks the chunks of expert e.
__global__ void __launch_bounds__(kMaxE) group_scan_kernel(MoEArgs a, const int* ccnt, int* coff,
                                                           int nchunks) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int s_tot[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_uoff[kMaxE + 1];
  const int E = a.E, e = threadIdx.x;
  int tot = 0;
  if (e < E)
    for (int c = 0; c < nchunks; ++c) tot += ldg_cg_i32(ccnt + (size_t)c * E + e);
  s_tot[e] = e < E ? tot : 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0, urun = 0;
    for (int i = 0; i < E; ++i) {
      s_off[i] = run;
      s_uoff[i] = urun;
      run += s_tot[i];
      urun += s_tot[i] > 0;
    }
    s_off[E] = run;
    s_uoff[E] = urun;
    a.ws.e_off[E] = run;
    a.ws.uniq[0] = urun;
  }
  __syncthreads();
  if (e < E) {
    a.ws.e_cnt[e] = s_tot[e];
    a.ws.e_off[e] = s_off[e];
    if (s_tot[e] > 0) a.ws.uniq[1 + s_uoff[e]] = e;
    int run = s_off[e];
    for (int c = 0; c < nchunks; ++c) {
      coff[(size_t)c * E + e] = run;
      run += ldg_cg_i32(ccnt + (size_t)c * E + e);
    }
  }
}

// Stable scatter of one chunk: pairs are taken in order, kGroupThreads at a
// time; the rank of a pair among equal experts of the same batch comes from
// __match_any_sync inside a warp plus per-warp counts across warps.
__global__ void __launch_bounds__(kGroupThreads) group_scatter_kernel(MoEArgs a, const int* coff,
                                                                      int* rowof) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int kW = kGroupThreads / 32;
  __shared__ int s_base[kMaxE];
  __shared__ int s_wcnt[kW][kMaxE];
  const int E = a.E, np = a.M * a.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_base[e] = ldg_cg_i32(coff + (size_t)blockIdx.x * E + e);
  const int p0 = blockIdx.x * kGroupChunk;
  for (int b = 0; b < kGroupChunk; b += kGroupThreads) {
    for (int i = threadIdx.x; i < kW * kMaxE; i += blockDim.x) (&s_wcnt[0][0])[i] = 0;
    __syncthreads();
    const int p = p0 + b + threadIdx.x;
    const int e = p < np ? ldg_cg_i32(a.ws.ids + p) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank_w = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank_w == 0) s_wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += s_wcnt[w][e];
      const int pos = s_base[e] + before + rank_w;
      a.ws.sorted_pairs[pos] = p;
      rowof[p] = pos;
    }
    __syncthreads();
    if (e >= 0 && rank_w == 0) {
      int tot = 0;
      for (int w = 0; w < kW; ++w) tot += s_wcnt[w][e];
      // one writer per expert per warp; only the first warp holding e adds
      bool first = true;
      for (int w = 0; w < warp; ++w) first = first && (s_wcnt[w][e] == 0);
      if (first) s_base[e] += tot;
    }
    __syncthreads();
  }
}

// ----------------------------------------------------------------------------
static cudaError_t launch(const void* fn, dim3 grid, dim3 block, void** args, cudaStream_t st,
                          bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_route(const MoEArgs& a, bool build_meta, cudaStream_t st, bool pdl) {
  int* rowof = a.ws.rowof;
  const bool small = a.M <= kDecodeMaxTokens;
  int meta_in_router = (build_meta && small) ? 1 : 0;
  MoEArgs aa = a;
  void* args[] = {&aa, &meta_in_router, &rowof};
  dim3 grid((a.E + kRouteWarps - 1) / kRouteWarps, (a.M + kRouteTokens - 1) / kRouteTokens);
  cudaError_t err = launch((const void*)route_kernel, grid, dim3(kRouteWarps * 32), args, st, pdl);
  if (err != cudaSuccess || !build_meta || small) return err;

  const int np = a.M * a.k;
  int nchunks = (np + kGroupChunk - 1) / kGroupChunk;
  int* ccnt = a.ws.gcnt;
  int* coff = a.ws.gcnt + (size_t)nchunks * a.E;
  void* a1[] = {&aa, &ccnt};
  err = launch((const void*)group_count_kernel, dim3(nchunks), dim3(kGroupThreads), a1, st, true);
  if (err != cudaSuccess) return err;
  void* a2[] = {&aa, &ccnt, &coff, &nchunks};
  err = launch((const void*)group_scan_kernel, dim3(1), dim3(kMaxE), a2, st, true);
  if (err != cudaSuccess) return err;
  void* a3[] = {&aa, &coff, &rowof};
  return launch((const void*)group_scatter_kernel, dim3(nchunks), dim3(kGroupThreads), a3, st, true);
}

}  // namespace flint
