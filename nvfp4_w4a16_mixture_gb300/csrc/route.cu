// Router GEMV + top-k + expert grouping.
//
// Router logits, top-k, sigmoid renormalisation: vLLM page
// "vllm.models.flint.ops.moe", _router_kernel / _topk_row docstrings (BF16
// logits, ties to the lowest expert index, s / (sum + 1e-20) rounded to
// BF16).  Expert grouping (histogram, exclusive scan, stable scatter of the
// (token, slot) pairs by expert) is the token permutation the grouped path of
// flint_moe consumes ("perm" of _combine_kernel); the decode path uses the
// same grouping to stream each routed expert's weights once per call.
#include <atomic>

#include <cooperative_groups.h>
#include <cuda_fp16.h>

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
    int* rec = a.ws.urec + (size_t)s_uoff[e] * kUrecInts;
    if (s_cnt[e] > 0) {
      a.ws.uniq[1 + s_uoff[e]] = e;
      rec[0] = e;
      rec[1] = s_cnt[e];
      rec[2] = s_off[e];
    }
    int c = s_off[e];
    for (int t = 0; t < M; ++t) {
      int j = s_pos[t][e];
      if (j != 0xFF) {
        int p = t * k + j;
        a.ws.sorted_pairs[c] = p;
        rowof[p] = c;
        rec[4 + c - s_off[e]] = p;
        ++c;
      }
    }
  }
  if (tid == 0) { a.ws.e_off[E] = s_off[E]; a.ws.uniq[0] = s_uoff[E]; }
}

// ----------------------------------------------------------------------------
// The fp32 router dot product of one token row with one router row in the
// canonical order (see route_kernel); `wreg` holds the row's 16-byte chunks
// when H <= 2048, else they are read from `wrow`.  Every lane returns the
// butterfly result (lane 0's value is the one that is rounded to BF16).
template <bool XSMEM = false>
FLINT_DEV float router_dot(const uint16_t* xrow, const uint4 (&wreg)[8], const uint16_t* wrow,
                           int H, int lane) {
  auto xload = [&](int h) {
    return XSMEM ? *reinterpret_cast<const uint4*>(xrow + h) : ldg_cg_v4(xrow + h);
  };
  const int nchunk = (H + 255) / 256;
  float acc = 0.0f;
  auto chunk = [&](const uint4& xv, const uint4& wv) {
    const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc = fmaf(__uint_as_float(xs[q] << 16), __uint_as_float(ws[q] << 16), acc);
      acc = fmaf(__uint_as_float(xs[q] & 0xFFFF0000u), __uint_as_float(ws[q] & 0xFFFF0000u), acc);
    }
  };
  if (H <= 2048) {
    // every chunk's load is issued before the first product, so the loads
    // overlap instead of costing one round trip each
    uint4 xreg[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int h = 256 * c + 8 * lane;
      xreg[c] = (c < nchunk && h < H) ? xload(h) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
      if (c < nchunk && 256 * c + 8 * lane < H) chunk(xreg[c], wreg[c]);
  } else {
    for (int c = 0; c < nchunk; ++c) {
      const int h = 256 * c + 8 * lane;
      if (h < H) chunk(xload(h), ldg_nc_v4(wrow + h));
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) acc = acc + __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// router_dot for a block of 4 experts x 2 NP tokens (H <= 2048): every
// (expert, token) chain is the same per-lane sequence of fp32 fmas (chunk c
// ascending, element k ascending) and the same butterfly; the 8 NP chains run
// side by side so that each x vector loaded from shared memory feeds four
// experts and each router vector 2 NP tokens.  Two tokens' chains share one
// packed fma.rn.f32x2 (two independent IEEE fmas), so the chains round
// exactly as scalar fmaf does.  x is in fp32 in shared memory, token pairs
// interleaved: pair p, chunk c, quad q (elements 2q, 2q + 1 of the lane's
// 8), lane l holds float4 {x[2p][h], x[2p + 1][h], x[2p][h + 1],
// x[2p + 1][h + 1]} with h = 256 c + 8 l + 2 q (kRtPairFloats floats per
// pair).  Experts e >= E read row E - 1 and are not stored by the caller.
constexpr int kRtPairFloats = 2 * 2048;

FLINT_DEV uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
FLINT_DEV void f32x2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
FLINT_DEV void fma_f32x2(uint64_t& acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// One 256-wide chunk of the block: w holds the lane's 8 router elements of
// the 4 experts, xc points at pair 0's chunk.
template <int NP>
FLINT_DEV void router_chunk(uint64_t (&acc)[4][NP], const uint4 (&w)[4], const float* xc, int lane) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    ulonglong2 xv[NP];  // per pair: {x(2q) of both tokens, x(2q + 1) of both tokens}
#pragma unroll
    for (int p = 0; p < NP; ++p)
      xv[p] = *reinterpret_cast<const ulonglong2*>(xc + (size_t)p * kRtPairFloats + (q * 32 + lane) * 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t word = q == 0 ? w[i].x : q == 1 ? w[i].y : q == 2 ? w[i].z : w[i].w;
      const float w0 = __uint_as_float(word << 16), w1 = __uint_as_float(word & 0xFFFF0000u);
      const uint64_t w0p = f32x2_pack(w0, w0), w1p = f32x2_pack(w1, w1);
#pragma unroll
      for (int p = 0; p < NP; ++p) fma_f32x2(acc[i][p], xv[p].x, w0p);
#pragma unroll
      for (int p = 0; p < NP; ++p) fma_f32x2(acc[i][p], xv[p].y, w1p);
    }
  }
}

template <int NP>
FLINT_DEV void router_block(float (&res)[4][2 * NP], const float* xp0, const uint16_t* router_w,
                            int e0, int E, int H, int lane) {
  const int nchunk = (H + 255) / 256;
  uint64_t acc[4][NP];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int p = 0; p < NP; ++p) acc[i][p] = 0ull;  // +0.0f in both halves
  const uint16_t* wr[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) wr[i] = router_w + (size_t)min(e0 + i, E - 1) * H + 8 * lane;
  auto load = [&](uint4 (&w)[4], int c) {
    const bool has = c < nchunk && 256 * c + 8 * lane < H;
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = has ? ldg_nc_v4(wr[i] + 256 * c) : make_uint4(0, 0, 0, 0);
  };
  // two register sets of router vectors, the next chunk's in flight
  uint4 wa[4], wb[4];
  load(wa, 0);
  for (int c = 0; c < nchunk; c += 2) {
    load(wb, c + 1);
    if (256 * c + 8 * lane < H) router_chunk<NP>(acc, wa, xp0 + (size_t)c * 512, lane);
    load(wa, c + 2);
    if (c + 1 < nchunk && 256 * (c + 1) + 8 * lane < H)
      router_chunk<NP>(acc, wb, xp0 + (size_t)(c + 1) * 512, lane);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      float v[2];
      f32x2_unpack(acc[i][p], v[0], v[1]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) v[h] = v[h] + __shfl_xor_sync(0xffffffffu, v[h], o);
        res[i][2 * p + h] = v[h];
      }
    }
}

FLINT_DEV void router_row_regs(uint4 (&wreg)[8], const uint16_t* wrow, int H, int lane, bool active) {
  const int nchunk = (H + 255) / 256;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    int h = 256 * c + 8 * lane;
    wreg[c] = (active && c < nchunk && h < H && H <= 2048) ? ldg_nc_v4(wrow + h) : make_uint4(0, 0, 0, 0);
  }
}

// Top-k of one token by one warp from its E BF16 logit bit patterns
// (get(e)): key = (order-preserving bf16 bits << 8) | (E - 1 - e), so the
// maximum key is the largest logit and, among equal bit patterns, the lowest
// expert index.  s = 1 / (1 + exp(-logit)) in fp32, summed in rank order;
// lane j < k ends with the j-th expert and tw = bf16(s_j / (sum + 1e-20)).
template <class Get>
FLINT_DEV void topk_warp(Get get, int E, int k, int lane, int& out_e, float& out_w) {
  int key[kMaxE / 32];
#pragma unroll
  for (int q = 0; q < kMaxE / 32; ++q) {
    int ee = q * 32 + lane;
    key[q] = -1;
    if (ee < E) key[q] = (int)((ordered_bf16(get(ee)) << 8) | (uint32_t)(E - 1 - ee));
  }
  int my_e = 0, my_key = 0;
  for (int j = 0; j < k; ++j) {  // selection only; lane j keeps rank j
    int lm = key[0];
#pragma unroll
    for (int q = 1; q < kMaxE / 32; ++q) lm = max(lm, key[q]);
    const int best = __reduce_max_sync(0xffffffffu, lm);
#pragma unroll
    for (int q = 0; q < kMaxE / 32; ++q)
      if (key[q] == best) key[q] = -1;
    if (lane == j) { my_key = best; my_e = E - 1 - (best & 0xFF); }
  }
  // the k sigmoids side by side, then their sum in rank order
  float my_s = 0.0f;
  if (lane < k) {
    const uint32_t o = (uint32_t)my_key >> 8;
    const uint32_t b16 = (o & 0x8000u) ? (o ^ 0x8000u) : (o ^ 0xFFFFu);
    const float logit = bf16_bits_to_f32(b16);
    my_s = __fdiv_rn(1.0f, 1.0f + expf(-logit));
  }
  float sum = 0.0f;
  for (int j = 0; j < k; ++j) sum = sum + __shfl_sync(0xffffffffu, my_s, j);
  out_e = my_e;
  out_w = round_bf16(__fdiv_rn(my_s, sum + 1e-20f));
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
  SpanGuard<kSpanRoute> span_guard;
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouteWarps + warp;
  const int tb = blockIdx.y;
  const int H = a.H, E = a.E, k = a.k;
  const int t0 = tb * kRouteTokens;
  const int nt = min(kRouteTokens, a.M - t0);
  const bool active = e < E;
  const uint16_t* wrow = a.router_w + (size_t)(active ? e : 0) * H;

  // router weights do not depend on earlier grids: fetch before the wait
  uint4 wreg[8];
  router_row_regs(wreg, wrow, H, lane, active);
  pdl_wait();

  if (active) {
    for (int tt = 0; tt < nt; ++tt) {
      const float acc = router_dot(a.x + (size_t)(t0 + tt) * H, wreg, wrow, H, lane);
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
    int my_e;
    float w;
    topk_warp([&](int ee) { return ldg_cg_u16(a.ws.logits + (size_t)t * E + ee); }, E, k, lane,
              my_e, w);
    if (lane < k) {
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
  SpanGuard<kSpanGroupCount> span_guard;
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
  SpanGuard<kSpanGroupScan> span_guard;
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
  SpanGuard<kSpanGroupScatter> span_guard;
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

// ----------------------------------------------------------------------------
// Router for few tokens (M <= kRcMaxTokens) as one cluster of kRcCtas CTAs:
// warp w of CTA r computes the logits of experts r * kRcWarps + w (+ multiples
// of kRcCtas * kRcWarps) for every token, with router_dot (the canonical
// order, so ids match route_kernel bit for bit), and stores them into the
// leader CTA's shared memory.  After the cluster barrier the other CTAs make
// the f16 copy of x for the gate/up kernel while the leader runs the top-k
// (warp per token) and the expert grouping from shared memory: per
// expert a bit mask of its tokens, counts and offsets by a scan, a pair's
// sorted position = its expert's offset + the number of earlier tokens in the
// mask.  No global atomics and no re-reads of global results on the way.
constexpr int kRcCtas = 8;
constexpr int kRcWarps = 16;
constexpr int kRcMaxTokens = 16;

struct RcSmem {
  uint16_t logit[kRcMaxTokens][kMaxE];
  int ids[kRcMaxTokens][kMaxTopK];
  unsigned long long mask[kMaxE];
  int off[kMaxE + 1];
  int uidx[kMaxE + 1];
};

__global__ void __cluster_dims__(kRcCtas, 1, 1) __launch_bounds__(kRcWarps * 32)
    route_cluster_kernel(MoEArgs a) {
  SpanGuard<kSpanRoute> span_guard;
  __shared__ RcSmem S;
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int H = a.H, E = a.E, k = a.k, M = a.M;
  RcSmem* lead = cl.map_shared_rank(&S, 0);

  // The first router row of this warp is a weight, independent of earlier
  // kernels: its load overlaps the previous kernel's tail.  Then wait for
  // that kernel (x may be its output), and only then let the gate/up kernel
  // start, because it reads x before its own dependency wait.
  const int e0 = rank * kRcWarps + warp;
  uint4 wreg[8];
  router_row_regs(wreg, a.router_w + (size_t)min(e0, E - 1) * H, H, lane, e0 < E);
  pdl_wait();
  pdl_launch_dependents();

  for (int e = e0; e < E; e += kRcCtas * kRcWarps) {
    const uint16_t* wrow = a.router_w + (size_t)e * H;
    if (e != e0) router_row_regs(wreg, wrow, H, lane, true);
    for (int t = 0; t < M; ++t) {
      const float acc = router_dot(a.x + (size_t)t * H, wreg, wrow, H, lane);
      if (lane == 0) lead->logit[t][e] = (uint16_t)f32_to_bf16_bits(acc);
    }
  }
  cl.sync();  // every logit is in the leader's shared memory
  if (rank != 0) {
    // f16 copy of x for the gate/up kernel, made by the other CTAs while the
    // leader runs the top-k: per token the power of two that puts the largest
    // magnitude in [2^14, 2^15); CTA r converts the column pairs
    // [(r - 1) P / (kRcCtas - 1), r P / (kRcCtas - 1)) of every token (P =
    // H / 2) and reports whether every value survived the round trip (then
    // the copy is exact)
    static_assert(kRcMaxTokens <= kX16MaxTokens, "the f16 copy covers the cluster router's tokens");
    __shared__ int s_exp[kRcMaxTokens];
    __shared__ int s_bad;
    if (tid == 0) s_bad = 0;
    for (int t = warp; t < M; t += kRcWarps) {
      uint32_t mx = 0;  // largest bf16 magnitude bit pattern (orders like the values)
      for (int h = 8 * lane; h < H; h += 256) {
        const uint4 v = ldg_cg_v4(a.x + (size_t)t * H + h);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
      }
      mx = __reduce_max_sync(0xffffffffu, mx);
      if (lane == 0) {
        int e = 0;
        if (mx >= 0x7F80u) e = 1000;  // inf or nan: no f16 copy
        else if (mx != 0) e = min(126, max(-110, 14 - ((int)(mx >> 7) - 127)));
        s_exp[t] = e;
      }
    }
    __syncthreads();
    const int P = H / 2, p0 = (rank - 1) * P / (kRcCtas - 1), p1 = rank * P / (kRcCtas - 1);
    const int np = p1 - p0;
    bool bad = false;
    for (int i = tid; i < M * np; i += kRcWarps * 32) {
      const int t = i / np, h = 2 * (p0 + i % np);
      const int e = s_exp[t];
      if (e == 1000) { bad = true; continue; }
      const uint32_t xv = *reinterpret_cast<const uint32_t*>(a.x + (size_t)t * H + h);
      const float sc = pow2f(e);
      const float f0 = __uint_as_float(xv << 16) * sc, f1 = __uint_as_float(xv & 0xFFFF0000u) * sc;
      const __half2 hv = __floats2half2_rn(f0, f1);
      const float2 back = __half22float2(hv);
      if (back.x != f0 || back.y != f1) bad = true;
      *reinterpret_cast<__half2*>(a.ws.x16 + (size_t)t * H + h) = hv;
    }
    if (bad) s_bad = 1;
    __syncthreads();
    if (tid == 0 && s_bad) atomicAdd(&a.ws.glob_cnt[1], 1);
    if (rank == 1 && tid < M) a.ws.x16_exp[tid] = s_exp[tid];
    return;
  }

  for (int e = tid; e < E; e += kRcWarps * 32) S.mask[e] = 0ull;
  for (int t = warp; t < M; t += kRcWarps) {
    int my_e;
    float w;
    topk_warp([&](int ee) { return (uint32_t)S.logit[t][ee]; }, E, k, lane, my_e, w);
    if (lane < k) {
      S.ids[t][lane] = my_e;
      a.ws.ids[t * k + lane] = my_e;
      a.ws.tw[t * k + lane] = w;
      if (a.ids_out) a.ids_out[t * k + lane] = my_e;
      if (a.tw_out) a.tw_out[t * k + lane] = w;
    }
  }
  __syncthreads();
  const int np = M * k;
  for (int p = tid; p < np; p += kRcWarps * 32)
    atomicOr(&S.mask[S.ids[p / k][p % k]], 1ull << (p / k));
  __syncthreads();
  if (warp == 0) {  // exclusive scans of counts and of "routed" flags
    // lane l takes experts per * l .. per * l + per - 1: its own sums, then
    // one warp scan of the lanes' totals
    constexpr int kPer = kMaxE / 32;
    const int per = (E + 31) / 32;
    int c[kPer], sc = 0, su = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = per * lane + q;
      c[q] = q < per && e < E ? __popcll(S.mask[e]) : 0;
      sc += c[q];
      su += c[q] > 0 ? 1 : 0;
    }
    int ic = sc, iu = su;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vc = __shfl_up_sync(0xffffffffu, ic, o);
      const int vu = __shfl_up_sync(0xffffffffu, iu, o);
      if (lane >= o) { ic += vc; iu += vu; }
    }
    int run = ic - sc, urun = iu - su;  // exclusive starts of this lane's experts
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = per * lane + q;
      if (q < per && e < E) {
        S.off[e] = run;
        S.uidx[e] = urun;
      }
      run += c[q];
      urun += c[q] > 0 ? 1 : 0;
    }
    if (lane == 31) { S.off[E] = ic; S.uidx[E] = iu; }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kRcWarps * 32) {
    const int c = __popcll(S.mask[e]);
    a.ws.e_cnt[e] = c;
    a.ws.e_off[e] = S.off[e];
    if (c > 0) {
      a.ws.uniq[1 + S.uidx[e]] = e;
      int* rec = a.ws.urec + (size_t)S.uidx[e] * kUrecInts;
      rec[0] = e;
      rec[1] = c;
      rec[2] = S.off[e];
    }
  }
  if (tid == 0) { a.ws.e_off[E] = S.off[E]; a.ws.uniq[0] = S.uidx[E]; }
  for (int p = tid; p < np; p += kRcWarps * 32) {
    const int t = p / k, e = S.ids[t][p % k];
    const int r = __popcll(S.mask[e] & ((1ull << t) - 1ull));
    const int pos = S.off[e] + r;
    a.ws.sorted_pairs[pos] = p;
    a.ws.rowof[p] = pos;
    a.ws.urec[(size_t)S.uidx[e] * kUrecInts + 4 + r] = p;
  }
}

// ----------------------------------------------------------------------------
// Router for many tokens: CTA b handles tokens 16 b .. 16 b + 15 with their
// rows staged in shared memory; the warps take blocks of 4 experts x 8 tokens
// (router_block, H <= 2048) or one expert's row for all 16 tokens
// (router_dot, longer rows), the canonical per-chain order either way, so ids
// match the other routers bit for bit; then warp w runs the top-k of token
// 16 b + w from shared memory.  No cross-CTA step.
constexpr int kRtTokens = 16;
constexpr int kRtWarps = 16;

__global__ void __launch_bounds__(kRtWarps * 32) route_tile_kernel(MoEArgs a) {
  SpanGuard<kSpanRoute> span_guard;
  extern __shared__ __align__(16) uint8_t rt_smem[];
  const int H = a.H, E = a.E, k = a.k;
  const bool f32 = H <= 2048;
  float* xf = reinterpret_cast<float*>(rt_smem);      // H <= 2048: [8 pairs][4096] fp32, pair order
  uint16_t* xs = reinterpret_cast<uint16_t*>(rt_smem);  // H > 2048: [16][H] bf16
  uint16_t* lg = reinterpret_cast<uint16_t*>(rt_smem + (f32 ? (size_t)kRtTokens * 2048 * 4
                                                             : (size_t)kRtTokens * H * 2));  // [16][E]
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRtTokens;
  const int nt = min(kRtTokens, a.M - t0);
  pdl_wait();
  {  // stage the token rows (16-byte vectors of 8 elements)
    const int nvr = H / 8;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)t0 * H);
    if (f32) {
      // vector v = h / 8 of tokens 2p and 2p + 1 -> pair p, chunk v / 32,
      // lane v % 32: four float4, one per quad of elements (tokens past nt
      // read as zero)
      const int np = (nt + 1) / 2, nv = np * nvr;
      for (int i = threadIdx.x; i < nv; i += blockDim.x) {
        const int p = i / nvr, v = i % nvr;
        const uint4 q0 = ldg_cg_v4(src + (size_t)(2 * p) * nvr + v);
        const uint4 q1 = 2 * p + 1 < nt ? ldg_cg_v4(src + (size_t)(2 * p + 1) * nvr + v)
                                        : make_uint4(0, 0, 0, 0);
        const uint32_t a0[4] = {q0.x, q0.y, q0.z, q0.w}, a1[4] = {q1.x, q1.y, q1.z, q1.w};
        float* d = xf + (size_t)p * kRtPairFloats + (v >> 5) * 512 + (v & 31) * 4;
#pragma unroll
        for (int qd = 0; qd < 4; ++qd)
          *reinterpret_cast<float4*>(d + qd * 128) =
              make_float4(__uint_as_float(a0[qd] << 16), __uint_as_float(a1[qd] << 16),
                          __uint_as_float(a0[qd] & 0xFFFF0000u), __uint_as_float(a1[qd] & 0xFFFF0000u));
      }
    } else {
      for (int i = threadIdx.x; i < nt * nvr; i += blockDim.x) reinterpret_cast<uint4*>(xs)[i] = ldg_cg_v4(src + i);
    }
  }
  __syncthreads();
  if (f32) {
    // blocks of 4 experts x 8 tokens; chains of tokens past nt run on stale
    // shared memory and are not stored
    const int neb = (E + 3) / 4, ntb = (nt + 7) / 8;
    for (int b = warp; b < neb * ntb; b += kRtWarps) {
      const int e0 = 4 * (b / ntb), tb = 8 * (b % ntb);
      float r[4][8];
      router_block<4>(r, xf + (size_t)(tb / 2) * kRtPairFloats, a.router_w, e0, E, H, lane);
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (e0 + i < E && tb + j < nt) lg[(tb + j) * E + e0 + i] = (uint16_t)f32_to_bf16_bits(r[i][j]);
      }
    }
  }
  for (int e = warp; e < E && !f32; e += kRtWarps) {
    const uint16_t* wrow = a.router_w + (size_t)e * H;
    uint4 wreg[8];
    router_row_regs(wreg, wrow, H, lane, true);
    {
      for (int t = 0; t < nt; ++t) {
        const float acc = router_dot<true>(xs + (size_t)t * H, wreg, wrow, H, lane);
        if (lane == 0) lg[t * E + e] = (uint16_t)f32_to_bf16_bits(acc);
      }
    }
  }
  __syncthreads();
  if (warp < nt) {
    const int t = t0 + warp;
    int my_e;
    float w;
    topk_warp([&](int ee) { return (uint32_t)lg[warp * E + ee]; }, E, k, lane, my_e, w);
    if (lane < k) {
      a.ws.ids[t * k + lane] = my_e;
      a.ws.tw[t * k + lane] = w;
      if (a.ids_out) a.ids_out[t * k + lane] = my_e;
      if (a.tw_out) a.tw_out[t * k + lane] = w;
    }
  }
}

size_t route_tile_smem(const MoEArgs& a) {
  return (a.H <= 2048 ? (size_t)kRtTokens * 2048 * 4 : (size_t)kRtTokens * a.H * 2) +
         (size_t)kRtTokens * a.E * 2;
}

bool route_cluster_supported(const MoEArgs& a) { return a.M <= kRcMaxTokens; }

cudaError_t launch_route_cluster(const MoEArgs& a, cudaStream_t st) {
  MoEArgs aa = a;
  void* args[] = {&aa};
  return launch((const void*)route_cluster_kernel, dim3(kRcCtas), dim3(kRcWarps * 32), args, st,
                true);
}

cudaError_t launch_route(const MoEArgs& a, bool build_meta, cudaStream_t st, bool pdl) {
  int* rowof = a.ws.rowof;
  const bool small = a.M <= kDecodeMaxTokens;
  int meta_in_router = (build_meta && small) ? 1 : 0;
  MoEArgs aa = a;
  void* args[] = {&aa, &meta_in_router, &rowof};
  cudaError_t err;
  if (!small && route_tile_smem(a) <= 200 * 1024) {
    static std::atomic<bool> attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
      err = cudaFuncSetAttribute((const void*)route_tile_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
      if (err != cudaSuccess) return err;
      attr_set[dev].store(true, std::memory_order_release);
    }
    void* targs[] = {&aa};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.M + kRtTokens - 1) / kRtTokens);
    cfg.blockDim = dim3(kRtWarps * 32);
    cfg.dynamicSmemBytes = route_tile_smem(a);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    err = cudaLaunchKernelExC(&cfg, (const void*)route_tile_kernel, targs);
  } else {
    dim3 grid((a.E + kRouteWarps - 1) / kRouteWarps, (a.M + kRouteTokens - 1) / kRouteTokens);
    err = launch((const void*)route_kernel, grid, dim3(kRouteWarps * 32), args, st, pdl);
  }
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

FLINT_SPAN_SETTER(route)

}  // namespace flint
