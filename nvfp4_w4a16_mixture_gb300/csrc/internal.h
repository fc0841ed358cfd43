// Internal interface between the C-ABI entry points and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "flint_moe.h"

namespace flint {

constexpr int kMaxE = 256;
constexpr int kMaxTopK = 32;
constexpr int kDecodeMaxTokens = 64;  // M above this uses the grouped path

// Offsets (bytes from the workspace base) of every workspace region, all
// 256-byte aligned.  The control block comes first: the status word and every
// counter, at offsets that depend only on (H, E, SI), with the per-token-block
// router counters last, so that a workspace sized for M serves any call with
// the same (H, E, I, SI) and a smaller M.  Every launch returns its counters
// to zero.  The data regions after it need no initial value.
struct WsLayout {
  size_t status;       // int32[4]: [0] first error recorded by a kernel
  size_t glob_cnt;     // int32[4]: global last-arriver counters
  size_t fd_cnt;       // int32[4]: single-launch decode grid barriers [0], [1], CTAs done [2]
  size_t hblk_cnt;     // int32[H / 16]: down/combine last-arriver counters
  size_t tok_cnt;      // int32[ceil(M / kRouteTokens)]: router last-arriver counters
  size_t logits;       // bf16 [M, E]
  size_t ids;          // int32 [M, k]
  size_t tw;           // fp32 [M, k]
  size_t e_cnt;        // int32 [E]: pairs routed to each expert
  size_t e_off;        // int32 [E + 1]: exclusive prefix of e_cnt
  size_t uniq;         // int32 [1 + E]: [0] = U (experts with >= 1 pair), then their ids
  size_t sorted_pairs; // int32 [M * k]: pair ids t*k+j, stable-sorted by expert
  size_t rowof;        // int32 [M * k]: sorted position of pair t*k+j
  size_t urec;         // int32 [min(E, M * k), kUrecInts]: per routed expert (M <= 64)
  size_t gcnt;         // int32 [2, nchunks, E]: per-chunk counts and offsets (grouping)
  size_t act;          // bf16 [M * k, I]   row = sorted position of the pair
  size_t sact;         // bf16 [M, SI]
  size_t y;            // bf16 [M * k, H]   row = sorted position of the pair
  size_t ys;           // bf16 [M, H]
  size_t x_perm;       // bf16 [M * k, H]: token rows in sorted pair order (grouped path)
  size_t st_table;     // int32 [entries, 4]: per-expert token tiles (grouped path)
  size_t st_count;     // int32: number of token tiles
  size_t x16;          // f16 [M, H]: x[t] * 2^x16_exp[t], exactly (M <= kX16MaxTokens)
  size_t x16_exp;      // int32 [M]
  size_t xn;           // bf16 [M, H]: normalised rows (add-RMSNorm entry point)
  size_t total;
};

// Few-token decode: the cluster router also writes each token's row as f16
// scaled by a power of two (the largest magnitude lands in [2^14, 2^15)) and
// counts, in glob_cnt[1], its CTAs that met a value the f16 copy does not hold
// exactly; the gate/up kernel uses the f16 copy only when that count is 0,
// and the down kernel returns the count to 0.
constexpr int kX16MaxTokens = 16;

constexpr int kRouteTokens = 8;  // tokens per router CTA
// Record of the u-th routed expert (M <= kDecodeMaxTokens): [0] expert id,
// [1] pairs routed to it, [2] sorted position of its first pair, [3] unused,
// [4 ..] its pair ids t * k + j in sorted order.
constexpr int kUrecInts = 4 + kDecodeMaxTokens;

WsLayout ws_layout(const flint_moe_shape& s);

struct Ws {  // device pointers into one workspace
  int* status;
  int* fd_cnt;
  int* tok_cnt;
  int* glob_cnt;
  int* hblk_cnt;
  uint16_t* logits;
  int* ids;
  float* tw;
  int* e_cnt;
  int* e_off;
  int* uniq;
  int* sorted_pairs;
  int* rowof;
  int* urec;
  uint16_t* x_perm;
  int* st_table;
  int* st_count;
  int* gcnt;
  uint16_t* act;
  uint16_t* sact;
  uint16_t* y;
  uint16_t* ys;
  uint16_t* x16;
  int* x16_exp;
  uint16_t* xn;
};

Ws ws_pointers(void* base, const WsLayout& L);

struct MoEArgs {
  const uint16_t* x;
  const uint16_t* router_w;
  const uint8_t* w13;
  const uint8_t* w13_sf;
  const float* w13_gs;
  const uint8_t* w2;
  const uint8_t* w2_sf;
  const float* w2_gs;
  const uint16_t* shared_gu;
  const uint16_t* shared_down;
  uint16_t* out;
  int* ids_out;   // optional user copy
  float* tw_out;  // optional user copy
  int M, H, E, k, I, SI;
  int fault;  // test hook: a FLINT_FAULT_* site whose signal is left out (0: none)
  Ws ws;
};

// The failure-path test hook's current site (flint_moe_debug_fault).
int debug_fault_site();

// Launchers (return cudaSuccess or the launch error).  `pdl` launches the
// kernel with programmatic stream serialisation.
cudaError_t launch_route(const MoEArgs& a, bool build_meta, cudaStream_t st, bool pdl);
// One-cluster router with the small-M grouping; for M <= 16.  Launched with
// programmatic dependent launch: it prefetches router rows, waits for the
// previous kernel, then releases its dependents.
bool route_cluster_supported(const MoEArgs& a);
cudaError_t launch_route_cluster(const MoEArgs& a, cudaStream_t st);
cudaError_t launch_decode_gate_up(const MoEArgs& a, cudaStream_t st, bool pdl);
cudaError_t launch_decode_down(const MoEArgs& a, cudaStream_t st, bool pdl);

// Grouped path of many tokens (tcgen05 GEMMs): router + grouping, plan,
// gather, GEMM1 (+ shared), GEMM2 (+ shared), combine.
bool grouped_supported(const flint_moe_shape& s);
size_t grouped_st_entries(const flint_moe_shape& s);
cudaError_t launch_grouped(const MoEArgs& a, cudaStream_t st);

// Decode path of few tokens: router, gate/up and down+combine kernels chained
// with programmatic dependent launch (M <= kDecodeMaxTokens and the limits
// decode2_supported checks).
bool decode2_supported(const flint_moe_shape& s);
cudaError_t launch_decode2(const MoEArgs& a, cudaStream_t st);

// Single-launch decode path (decode_fused.cu): router, top-k, grouping,
// gate/up, down and combine in one cooperative launch of `sms` CTAs, for
// M <= kFusedMaxTokens and the limits fused_supported checks.
constexpr int kFusedMaxTokens = 8;
bool fused_supported(const flint_moe_shape& s, int sms);
cudaError_t launch_fused(const MoEArgs& a, cudaStream_t st, int sms);

// norm.fused_add_rms_norm of rows a + r (add_norm.cu): residual' and xn, both
// bf16 [M, H]; one warp per token, launched with programmatic dependent launch.
cudaError_t launch_add_rms_norm(const uint16_t* a, const uint16_t* r, const uint16_t* w, float eps,
                                int M, int H, uint16_t* res_out, uint16_t* xn, cudaStream_t st);

// Kernel-span buffer setters, one per translation unit with kernels
// (flint_moe_record_spans calls them all).
cudaError_t span_buffer_set_decode2(unsigned long long* b);
cudaError_t span_buffer_set_decode(unsigned long long* b);
cudaError_t span_buffer_set_fused(unsigned long long* b);
cudaError_t span_buffer_set_grouped(unsigned long long* b);
cudaError_t span_buffer_set_route(unsigned long long* b);
cudaError_t span_buffer_set_add_norm(unsigned long long* b);
cudaError_t span_buffer_set_bf16_experts(unsigned long long* b);
cudaError_t span_buffer_set_shared_nvfp4(unsigned long long* b);
cudaError_t span_buffer_set_qkv(unsigned long long* b);

// NVFP4 shared expert (shared_nvfp4.cu): sact and ys (workspace), then
// out = bf16(out + ys) over the block's routed output.
cudaError_t launch_shared_nvfp4(const uint16_t* x, const uint8_t* gu, const uint8_t* gu_sf, const float* gu_gs,
                                const uint8_t* dn, const uint8_t* dn_sf, const float* dn_gs, int M, int H,
                                int SI, uint16_t* sact, uint16_t* ys, uint16_t* out, cudaStream_t st);

// Fused decode qkv (qkv.cu): the arguments of its GEMV and head kernels.
struct QkvArgs {
  int M, H, nq, nkv;
  const uint16_t* q_norm_w;
  const uint16_t* k_norm_w;
  float qk_eps;
  const float* cos_sin;  // [max_pos, 128] fp32 (cos | sin), or null: no RoPE
  long long max_pos;
  const long long* positions;     // [M]
  const long long* slot_mapping;  // [n_slots]
  int n_slots;
  uint16_t* k_cache;  // element offsets block * s_block + offset * s_slot + head * s_head + d
  uint16_t* v_cache;
  long long s_block, s_slot, s_head;
  int block_size;
  long long num_blocks;
  uint16_t* q_out;  // [M, nq * 128]
  uint16_t* xn;     // workspace [M, H]
  uint16_t* qkv;    // workspace [M, (nq + 2 nkv) * 128]
  int* status;      // workspace status word
};
// Input RMSNorm (add_norm.cu, residual may be null), the qkv GEMV (NVFP4 when
// w_sf is not null) and the head kernel.
cudaError_t launch_qkv_fused(const QkvArgs& a, const uint16_t* x, const uint16_t* residual,
                             const uint16_t* norm_w, float eps, const void* w, const uint8_t* w_sf,
                             const float* gs, uint16_t* res_out, cudaStream_t st);

// BF16 routed experts (bf16_experts.cu), M <= kDecodeMaxTokens: router with
// the expert grouping, exact gate/up and down sums, combine with the given
// shared output (null: none).
cudaError_t launch_bf16_experts(const MoEArgs& a, const uint16_t* w13, const uint16_t* w2,
                                const uint16_t* shared_out, cudaStream_t st);



}  // namespace flint
