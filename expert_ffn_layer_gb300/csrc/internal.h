// Kernel parameter blocks and launchers shared by the C ABI (api.cu) and the
// kernels.  Not part of the public interface.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------- router
struct RouterParams {
  CUtensorMap map_x;         // hidden [T][H] bf16, box {64, 128}, 128-byte swizzle
  CUtensorMap map_hi;        // W_high [E][H] bf16 (workspace), box {64, Epad}, 128-byte swizzle (rows >= E read 0)
  CUtensorMap map_lo;        // W_low, as map_hi
  __nv_bfloat16 *w_hi, *w_lo;  // [E][H] each, written by the split kernel
  float *partial;            // [KS][T][E] partial logits of the H slices
  const float *bias;         // [E] or nullptr
  float *logits_out;         // [T][E] or nullptr
  unsigned *err;             // workspace error word or nullptr
  int32_t *topk_idx;         // [T][k]
  float *topk_w;             // [T][k]
  int T, H, E, Epad, top_k, score_mode;
  float route_scale, renorm_eps;
  int kslices_per_cta;       // 64-wide K slices handled by one CTA
  int stages;
};
constexpr int kRouterThreads = 192;  // warp 0 TMA, 1 MMA, 2-5 epilogue
size_t router_smem_bytes(int Epad, int stages);
int router_stages(int Epad);
// split (router_w -> w_hi, w_lo), gemm (grid ksplit x mtiles), topk (grid T)
cudaError_t launch_router(const RouterParams &p, const float *router_w, int ksplit, int mtiles, cudaStream_t stream,
                          bool pdl);

// --------------------------------------------------------------- permute
struct PermuteParams {
  const int32_t *topk_idx;  // [S]
  int32_t *counts;          // [E]
  int32_t *offsets;         // [E + 1]
  int32_t *perm;            // [S]
  int32_t *inv;             // [S]
  unsigned *err;
  int32_t *part;            // [ceil(S / kPartSlots)][E] workspace table of the many-CTA path
  unsigned *done;           // workspace header word counting finished parts (left zero)
  int S, E;
};
// Batches above kPermuteOneCtaMax slots are permuted by ceil(S / kPartSlots)
// CTAs (count + scatter kernels); smaller ones by one CTA.
constexpr int kPartSlots = 1024;
constexpr int kPermuteOneCtaMax = 8192;
inline int permute_parts(int S) { return S > kPermuteOneCtaMax ? (S + kPartSlots - 1) / kPartSlots : 0; }
cudaError_t launch_permute(const PermuteParams &p, cudaStream_t stream, bool pdl);

// ------------------------------------------------------- grouped expert FFN
struct GemmParams {
  CUtensorMap map_wg, map_wu;  // w_gate, w_up {H, I, E}, box {64,128,1}
  CUtensorMap map_sg, map_su;  // ws_gate, ws_up {H, Is}, box {64,128}
  CUtensorMap map_wd;          // w_down {I, H, E}, box {64,128,1}
  CUtensorMap map_sd;          // ws_down {Is, H}, box {64,128}
  CUtensorMap map_act[4];      // A_act {I, S}, boxes {64, 16/32/64/128}
  CUtensorMap map_acts[4];     // A_shared {Is, T}, boxes {64, 16/32/64/128}
  const __nv_bfloat16 *hidden;  // [T][H], read row by row through perm
  const int32_t *perm;
  const int32_t *offsets;
  __nv_bfloat16 *act, *act_s;  // gate/up outputs: A_act [S][I], A_shared [T][Is]
  __nv_bfloat16 *y, *y_s;      // down outputs: y_sorted [S][H], y_shared [T][H]
  // mode 0: bf16 weights.  FP8 expert weights: the weight maps above are uint8
  // maps of E4M3 codes and sc_* the per-row fp32 scales; mode 1 (weight-only:
  // boxes {64, 128, 1}, no swizzle, expanded to bf16 in shared memory) or
  // mode 2 (W8A8: boxes {128, 128, 1}, 128-byte swizzle, FP8 MMAs on hq below)
  int mode;
  const float *sc_g, *sc_u, *sc_d;     // [E][I], [E][I], [E][H]
  const float *sc_sg, *sc_su, *sc_sd;  // [Is], [Is], [H]
  // W8A8 (mode 2): the hidden state quantised per token (codes [T][H], scales
  // [T]), and the gate/up epilogue's per-32-column maxima of the bf16
  // activations ([S][I/32] routed, [T][Is/32] shared) that set the down tiles'
  // per-row activation scales
  const uint8_t *hq;
  const float *hs;
  float *amax, *amax_s;
  // W8A8: the activations' E4M3 codes ([S][I], [T][Is]; map_act / map_acts then
  // describe these, boxes {128, 16/32/64/128}) and their per-row scales ([S], [T]),
  // written by the quantisation tiles
  uint8_t *aq, *aq_s;
  float *asc, *asc_s;
  unsigned *err;               // workspace error word
  unsigned *sync;              // workspace header: tile claim counter, exit counter, per-segment done counts
  int T, H, E, I, Is, top_k, S, has_shared;
  int phases;  // 1 gate/up only, 2 down only, 3 both (down tiles wait for their segment's gate/up tiles)
  // 1: the shared expert's first gate/up tiles start before the previous
  // kernel's results (perm, offsets) are awaited -- only when that kernel is
  // this library's permutation, in the layer chain
  int early;
  int gu_order;  // gate/up claim order: 1 level-major (row block outermost), 0 segment-major
};
// word offsets into the workspace header (4 KiB, zero when the workspace is fresh;
// every launch leaves them zero again)
constexpr int kSyncClaim = 64, kSyncExit = 65, kSyncPermute = 66,
              kSyncDone = 128,   // kSyncDone .. + 257: gate/up tiles finished, per segment
              kSyncQuant = 512;  // kSyncQuant .. + 257: W8A8 quantisation tiles finished, per segment
constexpr int kWsHeaderBytes = 4096;
int gemm_tile_n(int T, int top_k, int E);  // widest token tile (multiple of 16, <= 256) for a batch
cudaError_t launch_expert_ffn(const GemmParams &p, int bn, int num_ctas, cudaStream_t stream, bool pdl);

// --------------------------------------------------------------- combine
struct CombineParams {
  const __nv_bfloat16 *y_sorted;  // [S][H]
  const __nv_bfloat16 *y_shared;  // [T][H] or nullptr
  const int32_t *inv;             // [S]
  const float *topk_w;            // [T][k]
  __nv_bfloat16 *out;             // [T][H]
  int T, H, top_k, S;
};
cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream, bool pdl);

// ------------------------------------------------------------------- FP8
// codes [rows][cols] uint8 (E4M3) and scale [rows] fp32 of a bf16 [rows][cols]
// matrix, one scale per row; cols a multiple of 8, pointers 16-byte aligned
cudaError_t launch_quantize_rows(const __nv_bfloat16 *src, uint8_t *q, float *scale, long long rows, int cols,
                                 cudaStream_t stream);

// self-test: a bounded wait on a barrier nothing completes (records MOE_DEVERR_TIMEOUT)
cudaError_t launch_wait_timeout(unsigned *err, unsigned long long limit_ns, cudaStream_t stream);
// self-test: out[i] = the expert epilogue's SiLU(g[i]) * u[i], n >= 1
cudaError_t launch_silu_selftest(const float *g, const float *u, float *out, long long n, cudaStream_t stream);

// Unique id of the CUDA context current on the calling thread (0 when none is
// current yet).  Per-context state -- a kernel's shared-memory attribute, a
// module symbol's device address -- is cached under it rather than under the
// device ordinal: one ordinal names different contexts over a process's life
// (after cudaDeviceReset, or when a caller makes its own context current
// through the driver API).
unsigned long long context_id();
// cudaFuncSetAttribute(max dynamic shared memory) unless already done for the
// current context by this thread (done_ctx is the caller's per-thread cache).
cudaError_t set_smem_attr_once(const void *func, int bytes, unsigned long long &done_ctx);

// shared launch helper: PDL attribute on, optional cluster dims
cudaError_t launch_ex(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                      int cluster_x, void **args);

}  // namespace moe
