// C ABI (include/moe.h): argument validation, workspace layout, TMA tensor
// maps, and the launch chain.  Host code only; every step of the layer runs
// in the kernels of router.cu, permute.cu, expert_gemm.cu and combine.cu.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

cudaError_t launch_ex(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                      int cluster_x, void **args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = (unsigned)cluster_x;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = (unsigned)n;
  return cudaLaunchKernelExC(&cfg, func, args);
}

unsigned long long context_id() {
  using GetCurrent = CUresult (*)(CUcontext *);
  using GetId = CUresult (*)(CUcontext, unsigned long long *);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

cudaError_t set_smem_attr_once(const void *func, int bytes, unsigned long long &done_ctx) {
  const unsigned long long ctx = context_id();
  if (ctx != 0 && ctx == done_ctx) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  // the call above makes the primary context current if none was: look again
  if (e == cudaSuccess) done_ctx = ctx != 0 ? ctx : context_id();
  return e;
}

namespace {

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *ptr, const uint64_t *dims,
            const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const uint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void *>(ptr), (const cuuint64_t *)dims,
                  (const cuuint64_t *)strides_bytes, (const cuuint32_t *)box, (const cuuint32_t *)estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 matrix [rows][cols] row-major, box {64 cols, box_rows}, 128-byte swizzle
bool map_bf16_2d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t str[1] = {cols * 2};
  const uint32_t box[2] = {64, box_rows};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// E4M3 codes [rows][cols] (uint8), box {64 codes, box_rows}, no swizzle
bool map_u8_2d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t str[1] = {cols};
  const uint32_t box[2] = {64, box_rows};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ptr, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}
// stacked E4M3 codes [n][rows][cols], box {64, box_rows, 1}, no swizzle
bool map_u8_3d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint64_t n, uint32_t box_rows) {
  const uint64_t dims[3] = {cols, rows, n};
  const uint64_t str[2] = {cols, cols * rows};
  const uint32_t box[3] = {64, box_rows, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, ptr, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}
// E4M3 codes for the W8A8 kernel: boxes of 128 codes x box_rows, 128-byte
// swizzle (one 128-byte K-step row per matrix row, as the bf16 maps)
bool map_u8_2d_sw(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t str[1] = {cols};
  const uint32_t box[2] = {128, box_rows};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ptr, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
bool map_u8_3d_sw(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint64_t n, uint32_t box_rows) {
  const uint64_t dims[3] = {cols, rows, n};
  const uint64_t str[2] = {cols, cols * rows};
  const uint32_t box[3] = {128, box_rows, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, ptr, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// stacked bf16 [n][rows][cols] (consecutive matrices `stride_rows` rows apart,
// rows by default), box {64, box_rows, 1}, 128-byte swizzle
bool map_bf16_3d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint64_t n, uint32_t box_rows,
                 uint64_t stride_rows = 0) {
  const uint64_t dims[3] = {cols, rows, n};
  const uint64_t str[2] = {cols * 2, cols * (stride_rows ? stride_rows : rows) * 2};
  const uint32_t box[3] = {64, box_rows, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// ------------------------------------------------------------ validation
inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
inline bool aligned256(const void *p) { return ((uintptr_t)p & 255u) == 0; }
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
  size_t err, topk_idx, topk_w, counts, offsets, perm, inv, perm_part, y_sorted, y_shared, a_act, a_shared, w_hi,
      w_lo, partial, hq, hs, amax, amax_s, aq, aq_s, asc, asc_s, total;
};

// Split of H across router CTAs: a power of two <= 32 dividing H/64, with
// ksplit x (T/128 tiles) about the SM count.  With nsm = 256 it bounds every
// device's choice, which sizes the workspace without a device query.
int router_ksplit(const moe_dims &d, int nsm) {
  const int mtiles = (d.T + 127) / 128;
  const int nslices = d.H / 64;
  int ks = 32;
  while (ks > 1 && ((long long)mtiles * ks > nsm || nslices % ks != 0)) ks >>= 1;
  return ks;
}

WsLayout ws_layout(const moe_dims &d) {
  WsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t T = (size_t)d.T, S = (size_t)d.T * d.top_k, E = (size_t)d.E;
  const size_t Is = d.has_shared ? (size_t)d.I_shared : 0;
  L.err = take(kWsHeaderBytes);  // error word + tile-scheduler counters
  L.topk_idx = take(S * 4);
  L.topk_w = take(S * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm = take(S * 4);
  L.inv = take(S * 4);
  L.perm_part = take((size_t)permute_parts((int)S) * E * 4);
  L.y_sorted = take(S * (size_t)d.H * 2);
  L.y_shared = take(d.has_shared ? T * (size_t)d.H * 2 : 0);
  L.a_act = take(S * (size_t)d.I * 2);
  L.a_shared = take(T * Is * 2);
  L.w_hi = take(E * (size_t)d.H * 2);
  L.w_lo = take(E * (size_t)d.H * 2);
  L.partial = take((size_t)router_ksplit(d, 256) * T * E * 4);
  // W8A8: the hidden state's E4M3 codes and scales, and the activations' row maxima per 32 columns
  L.hq = take(T * (size_t)d.H);
  L.hs = take(T * 4);
  L.amax = take(S * (size_t)(d.I / 32) * 4);
  L.amax_s = take(T * (size_t)(Is / 32) * 4);
  // W8A8: the activations' E4M3 codes and their per-row scales (the quantisation tiles' output)
  L.aq = take(S * (size_t)d.I);
  L.aq_s = take(T * Is);
  L.asc = take(S * 4);
  L.asc_s = take(T * 4);
  L.total = off;
  return L;
}

int num_sms() {
  static thread_local int dev_cached = -1, n = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != dev_cached) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    dev_cached = dev;
  }
  return n > 0 ? n : 1;
}

inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <typename T>
inline T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

moe_status check_ws(const moe_dims *d, void *ws, size_t ws_bytes) {
  if (ws == nullptr || !aligned256(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_layout(*d).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// ------------------------------------------------------------ stages
moe_status do_route(const moe_dims &d, const moe_bf16 *hidden, const float *router_w, const float *bias,
                    float *logits_out, int32_t *topk_idx, float *topk_w, void *ws, cudaStream_t stream, bool pdl) {
  const WsLayout L = ws_layout(d);
  RouterParams p;
  std::memset(&p, 0, sizeof(p));
  const int Epad = (d.E + 15) & ~15;
  p.w_hi = at<__nv_bfloat16>(ws, L.w_hi);
  p.w_lo = at<__nv_bfloat16>(ws, L.w_lo);
  p.partial = at<float>(ws, L.partial);
  p.err = at<unsigned>(ws, L.err);
  if (!map_bf16_2d(&p.map_x, hidden, (uint64_t)d.H, (uint64_t)d.T, 128) ||
      !map_bf16_2d(&p.map_hi, p.w_hi, (uint64_t)d.H, (uint64_t)d.E, (uint32_t)Epad) ||
      !map_bf16_2d(&p.map_lo, p.w_lo, (uint64_t)d.H, (uint64_t)d.E, (uint32_t)Epad))
    return MOE_ERR_CUDA;
  p.bias = d.score_mode == MOE_SCORE_SIGMOID_BIAS ? bias : nullptr;
  p.logits_out = logits_out;
  p.topk_idx = topk_idx;
  p.topk_w = topk_w;
  p.T = d.T;
  p.H = d.H;
  p.E = d.E;
  p.Epad = Epad;
  p.top_k = d.top_k;
  p.score_mode = d.score_mode;
  p.route_scale = d.route_scale;
  p.renorm_eps = d.renorm_eps;
  p.stages = router_stages(Epad);
  const int mtiles = (d.T + 127) / 128;
  const int ks = router_ksplit(d, num_sms());
  p.kslices_per_cta = (d.H / 64) / ks;
  return cuda_status(launch_router(p, router_w, ks, mtiles, stream, pdl));
}

moe_status do_permute(const moe_dims &d, const int32_t *topk_idx, int32_t *counts, int32_t *offsets, int32_t *perm,
                      int32_t *inv, void *ws, cudaStream_t stream, bool pdl) {
  const WsLayout L = ws_layout(d);
  PermuteParams p;
  p.topk_idx = topk_idx;
  p.err = at<unsigned>(ws, L.err);
  p.done = at<unsigned>(ws, L.err) + kSyncPermute;
  p.part = at<int32_t>(ws, L.perm_part);
  p.counts = counts;
  p.offsets = offsets;
  p.perm = perm;
  p.inv = inv;
  p.S = d.T * d.top_k;
  p.E = d.E;
  return cuda_status(launch_permute(p, stream, pdl));
}

// The expert kernel's scratch: the workspace header (error word, tile-claim and
// completion counters) and the bf16 activations between gate/up and down.
struct ExpertScratch {
  unsigned *hdr;
  __nv_bfloat16 *act, *act_s;
  uint8_t *hq = nullptr;  // W8A8 only: the quantised hidden state and the activations' row maxima,
  float *hs = nullptr, *amax = nullptr, *amax_s = nullptr;
  uint8_t *aq = nullptr, *aq_s = nullptr;  // and the activations' codes and row scales
  float *asc = nullptr, *asc_s = nullptr;
};

// the scratch inside a caller's workspace (moe_workspace_bytes layout)
ExpertScratch scratch_in(const moe_dims &d, void *ws) {
  const WsLayout L = ws_layout(d);
  ExpertScratch sc;
  sc.hdr = at<unsigned>(ws, L.err);
  sc.act = at<__nv_bfloat16>(ws, L.a_act);
  sc.act_s = at<__nv_bfloat16>(ws, L.a_shared);
  sc.hq = at<uint8_t>(ws, L.hq);
  sc.hs = at<float>(ws, L.hs);
  sc.amax = at<float>(ws, L.amax);
  sc.amax_s = at<float>(ws, L.amax_s);
  sc.aq = at<uint8_t>(ws, L.aq);
  sc.aq_s = at<uint8_t>(ws, L.aq_s);
  sc.asc = at<float>(ws, L.asc);
  sc.asc_s = at<float>(ws, L.asc_s);
  return sc;
}

// Tensor maps and pointers of the grouped expert FFN; `phases` selects gate/up
// (1), down (2) or both in one persistent launch (3).  gu_stride: rows from one
// expert's gate (up) matrix to the next's -- I for separate [E, I, H] tensors,
// 2I when w_gate and w_up point into one [E, 2I, H] tensor (up = gate + I rows).
moe_status do_expert_phases(const moe_dims &d, int phases, const moe_bf16 *hidden, const int32_t *perm,
                            const int32_t *offsets, const moe_bf16 *w_gate, const moe_bf16 *w_up,
                            const moe_bf16 *w_down, const moe_bf16 *ws_gate, const moe_bf16 *ws_up,
                            const moe_bf16 *ws_down, moe_bf16 *y_sorted, moe_bf16 *y_shared,
                            const ExpertScratch &sc, cudaStream_t stream, bool pdl, uint64_t gu_stride = 0,
                            const moe_fp8_experts *q = nullptr, bool early = false, bool w8a8 = false) {
  // tiles of one launch at the narrowest chunking (16 tokens), for the 32-bit
  // claim counter and tile numbers
  {
    const long long S = (long long)d.T * d.top_k, Is = d.has_shared ? d.I_shared : 0;
    const long long rd = (d.H + 255) / 256;
    const long long worst = (S / 16 + d.E + 1) * ((d.I + 127) / 128 + rd) +
                            (d.has_shared ? (d.T / 16 + 1) * ((Is + 127) / 128 + rd) : 0);
    if (worst >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  }
  const int bn = gemm_tile_n(d.T, d.top_k, d.E);
  GemmParams g;
  std::memset(&g, 0, sizeof(g));
  g.T = d.T;
  g.H = d.H;
  g.E = d.E;
  g.I = d.I;
  g.Is = d.has_shared ? d.I_shared : 0;
  g.top_k = d.top_k;
  g.S = d.T * d.top_k;
  g.has_shared = d.has_shared;
  g.phases = phases;
  g.early = early && phases == 3 ? 1 : 0;
  // level-major gate/up order for batches whose experts average at most 256
  // tokens (weight streaming and MMAs overlap across SMs); segment-major for
  // the widest tiles (token rows stay hot in L2 across an expert's row blocks)
  g.gu_order = bn == 256 ? 0 : 1;
  g.hidden = reinterpret_cast<const __nv_bfloat16 *>(hidden);
  g.perm = perm;
  g.offsets = offsets;
  g.err = sc.hdr;
  g.sync = sc.hdr;
  g.act = sc.act;
  g.act_s = sc.act_s;
  g.y = reinterpret_cast<__nv_bfloat16 *>(y_sorted);
  g.y_s = reinterpret_cast<__nv_bfloat16 *>(y_shared);
  bool ok = true;
  if (q != nullptr && w8a8) {  // W8A8: swizzled code maps, the quantised hidden state, the row maxima
    g.mode = 2;
    g.sc_g = q->gate_scale;
    g.sc_u = q->up_scale;
    g.sc_d = q->down_scale;
    g.sc_sg = q->s_gate_scale;
    g.sc_su = q->s_up_scale;
    g.sc_sd = q->s_down_scale;
    g.hq = sc.hq;
    g.hs = sc.hs;
    g.amax = sc.amax;
    g.amax_s = sc.amax_s;
    g.aq = sc.aq;
    g.aq_s = sc.aq_s;
    g.asc = sc.asc;
    g.asc_s = sc.asc_s;
    ok = map_u8_3d_sw(&g.map_wg, q->gate, d.H, d.I, d.E, 128) && map_u8_3d_sw(&g.map_wu, q->up, d.H, d.I, d.E, 128) &&
         map_u8_3d_sw(&g.map_wd, q->down, d.I, d.H, d.E, 128);
    if (d.has_shared)
      ok = ok && map_u8_2d_sw(&g.map_sg, q->s_gate, d.H, g.Is, 128) &&
           map_u8_2d_sw(&g.map_su, q->s_up, d.H, g.Is, 128) && map_u8_2d_sw(&g.map_sd, q->s_down, g.Is, d.H, 128);
    // the down tiles load the activations' codes (128-code K steps) by TMA
    for (int b = 0; b < 4; ++b) ok = ok && map_u8_2d_sw(&g.map_act[b], g.aq, d.I, g.S, 16u << b);
    if (d.has_shared)
      for (int b = 0; b < 4; ++b) ok = ok && map_u8_2d_sw(&g.map_acts[b], g.aq_s, g.Is, d.T, 16u << b);
    if (!ok) return MOE_ERR_CUDA;
    return cuda_status(launch_expert_ffn(g, bn, num_sms(), stream, pdl));
  }
  if (q != nullptr) {  // FP8 expert weights: maps of the codes, and the row scales
    g.mode = 1;
    g.sc_g = q->gate_scale;
    g.sc_u = q->up_scale;
    g.sc_d = q->down_scale;
    g.sc_sg = q->s_gate_scale;
    g.sc_su = q->s_up_scale;
    g.sc_sd = q->s_down_scale;
    ok = map_u8_3d(&g.map_wg, q->gate, d.H, d.I, d.E, 128) && map_u8_3d(&g.map_wu, q->up, d.H, d.I, d.E, 128) &&
         map_u8_3d(&g.map_wd, q->down, d.I, d.H, d.E, 128);
    if (d.has_shared)
      ok = ok && map_u8_2d(&g.map_sg, q->s_gate, d.H, g.Is, 128) && map_u8_2d(&g.map_su, q->s_up, d.H, g.Is, 128) &&
           map_u8_2d(&g.map_sd, q->s_down, g.Is, d.H, 128);
    for (int b = 0; b < 4; ++b) ok = ok && map_bf16_2d(&g.map_act[b], g.act, d.I, g.S, 16u << b);
    if (d.has_shared)
      for (int b = 0; b < 4; ++b) ok = ok && map_bf16_2d(&g.map_acts[b], g.act_s, g.Is, d.T, 16u << b);
    if (!ok) return MOE_ERR_CUDA;
    return cuda_status(launch_expert_ffn(g, bn, num_sms(), stream, pdl));
  }
  if (phases & 1) {
    ok = ok && map_bf16_3d(&g.map_wg, w_gate, d.H, d.I, d.E, 128, gu_stride) &&
         map_bf16_3d(&g.map_wu, w_up, d.H, d.I, d.E, 128, gu_stride);
    if (d.has_shared)
      ok = ok && map_bf16_2d(&g.map_sg, ws_gate, d.H, g.Is, 128) && map_bf16_2d(&g.map_su, ws_up, d.H, g.Is, 128);
  }
  if (phases & 2) {
    ok = ok && map_bf16_3d(&g.map_wd, w_down, d.I, d.H, d.E, 128);
    for (int b = 0; b < 4; ++b) ok = ok && map_bf16_2d(&g.map_act[b], g.act, d.I, g.S, 16u << b);
    if (d.has_shared) {
      ok = ok && map_bf16_2d(&g.map_sd, ws_down, g.Is, d.H, 128);
      for (int b = 0; b < 4; ++b) ok = ok && map_bf16_2d(&g.map_acts[b], g.act_s, g.Is, d.T, 16u << b);
    }
  }
  if (!ok) return MOE_ERR_CUDA;
  return cuda_status(launch_expert_ffn(g, bn, num_sms(), stream, pdl));
}

// a5-a6: gate/up GEMM through the route index + SiLU(gate) * up -> activations in ws
moe_status do_gate_up(const moe_dims &d, const moe_bf16 *hidden, const int32_t *perm, const int32_t *offsets,
                      const moe_bf16 *w_gate, const moe_bf16 *w_up, const moe_bf16 *ws_gate, const moe_bf16 *ws_up,
                      void *ws, cudaStream_t stream, bool pdl) {
  return do_expert_phases(d, 1, hidden, perm, offsets, w_gate, w_up, nullptr, ws_gate, ws_up, nullptr, nullptr,
                          nullptr, scratch_in(d, ws), stream, pdl);
}

// a7-a8: down GEMM over the activations in ws -> y_sorted, y_shared
moe_status do_down(const moe_dims &d, const int32_t *offsets, const moe_bf16 *w_down, const moe_bf16 *ws_down,
                   moe_bf16 *y_sorted, moe_bf16 *y_shared, void *ws, cudaStream_t stream, bool pdl) {
  return do_expert_phases(d, 2, nullptr, nullptr, offsets, nullptr, nullptr, w_down, nullptr, nullptr, ws_down,
                          y_sorted, y_shared, scratch_in(d, ws), stream, pdl);
}

// a5-a8 in one persistent launch
moe_status do_expert_ffn(const moe_dims &d, const moe_bf16 *hidden, const int32_t *perm, const int32_t *offsets,
                         const moe_bf16 *w_gate, const moe_bf16 *w_up, const moe_bf16 *w_down,
                         const moe_bf16 *ws_gate, const moe_bf16 *ws_up, const moe_bf16 *ws_down, moe_bf16 *y_sorted,
                         moe_bf16 *y_shared, void *ws, cudaStream_t stream, bool pdl, bool early = false) {
  return do_expert_phases(d, 3, hidden, perm, offsets, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, y_sorted,
                          y_shared, scratch_in(d, ws), stream, pdl, 0, nullptr, early);
}

moe_status do_combine(const moe_dims &d, const moe_bf16 *y_sorted, const moe_bf16 *y_shared, const int32_t *inv,
                      const float *topk_w, moe_bf16 *out, cudaStream_t stream, bool pdl) {
  CombineParams c;
  c.y_sorted = reinterpret_cast<const __nv_bfloat16 *>(y_sorted);
  c.y_shared = d.has_shared ? reinterpret_cast<const __nv_bfloat16 *>(y_shared) : nullptr;
  c.inv = inv;
  c.topk_w = topk_w;
  c.out = reinterpret_cast<__nv_bfloat16 *>(out);
  c.T = d.T;
  c.H = d.H;
  c.top_k = d.top_k;
  c.S = d.T * d.top_k;
  return cuda_status(launch_combine(c, stream, pdl));
}

bool ptr_ok(const void *p) { return p != nullptr && aligned16(p); }

bool fp8_ok(const moe_dims &d, const moe_fp8_experts *q) {
  if (q == nullptr || !ptr_ok(q->gate) || !ptr_ok(q->up) || !ptr_ok(q->down) || !ptr_ok(q->gate_scale) ||
      !ptr_ok(q->up_scale) || !ptr_ok(q->down_scale))
    return false;
  if (d.has_shared && (!ptr_ok(q->s_gate) || !ptr_ok(q->s_up) || !ptr_ok(q->s_down) || !ptr_ok(q->s_gate_scale) ||
                       !ptr_ok(q->s_up_scale) || !ptr_ok(q->s_down_scale)))
    return false;
  return true;
}

// Steps a3-a9 from a given routing, with the gate and up projections of every
// expert stacked in one tensor: permutation, grouped expert FFN, combine.
moe_status do_fused_moe(const moe_dims &d, const moe_bf16 *hidden, const int32_t *topk_idx, const float *topk_w,
                        const moe_bf16 *w_gate_up, const moe_bf16 *w_down, const moe_bf16 *ws_gate_up,
                        const moe_bf16 *ws_down, moe_bf16 *out, void *ws, cudaStream_t s) {
  const WsLayout L = ws_layout(d);
  int32_t *perm = at<int32_t>(ws, L.perm), *inv = at<int32_t>(ws, L.inv);
  int32_t *offs = at<int32_t>(ws, L.offsets);
  moe_bf16 *y = at<moe_bf16>(ws, L.y_sorted), *z = at<moe_bf16>(ws, L.y_shared);
  moe_status st = do_permute(d, topk_idx, at<int32_t>(ws, L.counts), offs, perm, inv, ws, s, true);
  if (st != MOE_OK) return st;
  const size_t up = (size_t)d.I * d.H, sup = d.has_shared ? (size_t)d.I_shared * d.H : 0;
  st = do_expert_phases(d, 3, hidden, perm, offs, w_gate_up, w_gate_up + up, w_down, ws_gate_up,
                        d.has_shared ? ws_gate_up + sup : nullptr, ws_down, y, z, scratch_in(d, ws), s, true,
                        2 * (uint64_t)d.I, nullptr, true);
  if (st != MOE_OK) return st;
  return do_combine(d, y, z, inv, topk_w, out, s, true);
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API const char *moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null or misaligned pointer, bad size or mode";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape outside the supported set";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace smaller than moe_workspace_bytes()";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA launch or driver call failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a bounded wait inside a kernel ran out";
    case MOE_ERR_DEVICE_INDEX: return "MOE_ERR_DEVICE_INDEX: an index seen on the device was out of range";
  }
  return "unknown moe_status";
}

MOE_API moe_status moe_check_dims(const moe_dims *d) {
  if (d == nullptr) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->H <= 0 || d->E <= 0 || d->I <= 0 || d->top_k <= 0) return MOE_ERR_INVALID_ARG;
  if (d->has_shared != 0 && d->has_shared != 1) return MOE_ERR_INVALID_ARG;
  if (d->has_shared && d->I_shared <= 0) return MOE_ERR_INVALID_ARG;
  if (d->score_mode != MOE_SCORE_SIGMOID_BIAS && d->score_mode != MOE_SCORE_SOFTMAX) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(d->route_scale) || !std::isfinite(d->renorm_eps) || d->renorm_eps < 0.0f)
    return MOE_ERR_INVALID_ARG;
  if (d->score_mode == MOE_SCORE_SOFTMAX && d->route_scale != 1.0f) return MOE_ERR_INVALID_ARG;
  if (d->H % 64 != 0 || d->I % 64 != 0 || d->H > 16384 || d->I > 16384) return MOE_ERR_UNSUPPORTED;
  if (d->has_shared && (d->I_shared % 64 != 0 || d->I_shared > 16384)) return MOE_ERR_UNSUPPORTED;
  if (d->E > 256 || d->top_k > d->E || d->top_k > 16) return MOE_ERR_UNSUPPORTED;
  if ((long long)d->T * d->top_k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

MOE_API size_t moe_workspace_bytes(const moe_dims *d) {
  if (moe_check_dims(d) != MOE_OK) return 0;
  return ws_layout(*d).total;
}

MOE_API moe_status moe_ws_init(void *ws, size_t ws_bytes, void *stream) {
  if (ws == nullptr || !aligned256(ws) || ws_bytes < (size_t)kWsHeaderBytes) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, kWsHeaderBytes, (cudaStream_t)stream));
}

MOE_API moe_status moe_ws_read_error(void *ws, size_t ws_bytes, int clear, void *stream, uint32_t *bits) {
  if (ws == nullptr || !aligned256(ws) || ws_bytes < 256 || bits == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  *bits = v;
  return MOE_OK;
}

MOE_API moe_status moe_selftest_wait_timeout(void *ws, size_t ws_bytes, unsigned long long limit_ns, void *stream) {
  if (ws == nullptr || !aligned256(ws) || ws_bytes < 256) return MOE_ERR_INVALID_ARG;
  if (limit_ns == 0 || limit_ns > 10000000000ull) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_wait_timeout(at<unsigned>(ws, 0), limit_ns, (cudaStream_t)stream));
}

MOE_API moe_status moe_selftest_silu(const float *g, const float *u, float *out, int64_t n, void *stream) {
  if (n < 0) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  auto f32_ok = [](const float *p) { return p != nullptr && ((uintptr_t)p & 3u) == 0; };
  if (!f32_ok(g) || !f32_ok(u) || !f32_ok(out)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_silu_selftest(g, u, out, (long long)n, (cudaStream_t)stream));
}

MOE_API moe_status moe_route(const moe_dims *d, const moe_bf16 *hidden, const float *router_w,
                             const float *expert_bias, float *logits_out, int32_t *topk_idx, float *topk_w, void *ws,
                             size_t ws_bytes, void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;  // empty batch: T-sized buffers may be empty
  if (!ptr_ok(hidden) || !ptr_ok(router_w) || !ptr_ok(topk_idx) || !ptr_ok(topk_w)) return MOE_ERR_INVALID_ARG;
  if ((expert_bias != nullptr && !aligned16(expert_bias)) || (logits_out != nullptr && !aligned16(logits_out)))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != MOE_OK) return st;
  return do_route(*d, hidden, router_w, expert_bias, logits_out, topk_idx, topk_w, ws, (cudaStream_t)stream, true);
}

MOE_API moe_status moe_permute(const moe_dims *d, const int32_t *topk_idx, int32_t *counts, int32_t *offsets,
                               int32_t *perm, int32_t *inv_perm, void *ws, size_t ws_bytes, void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (!ptr_ok(counts) || !ptr_ok(offsets)) return MOE_ERR_INVALID_ARG;
  if (d->T > 0 && (!ptr_ok(topk_idx) || !ptr_ok(perm) || !ptr_ok(inv_perm))) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != MOE_OK) return st;
  if (d->T == 0) {
    // empty batch: counts and offsets are all zero
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(counts, 0, (size_t)d->E * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, (size_t)(d->E + 1) * 4, s);
    return cuda_status(e);
  }
  return do_permute(*d, topk_idx, counts, offsets, perm, inv_perm, ws, (cudaStream_t)stream, true);
}

MOE_API moe_status moe_expert_ffn(const moe_dims *d, const moe_bf16 *hidden, const int32_t *perm,
                                  const int32_t *offsets, const moe_bf16 *w_gate, const moe_bf16 *w_up,
                                  const moe_bf16 *w_down, const moe_bf16 *ws_gate, const moe_bf16 *ws_up,
                                  const moe_bf16 *ws_down, moe_bf16 *y_sorted, moe_bf16 *y_shared, void *ws,
                                  size_t ws_bytes, void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;
  if (!ptr_ok(hidden) || !ptr_ok(perm) || !ptr_ok(offsets) || !ptr_ok(w_gate) || !ptr_ok(w_up) || !ptr_ok(w_down) ||
      !ptr_ok(y_sorted))
    return MOE_ERR_INVALID_ARG;
  if (d->has_shared && (!ptr_ok(ws_gate) || !ptr_ok(ws_up) || !ptr_ok(ws_down) || !ptr_ok(y_shared)))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != MOE_OK) return st;
  return do_expert_ffn(*d, hidden, perm, offsets, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, y_sorted, y_shared,
                       ws, (cudaStream_t)stream, true);
}

MOE_API moe_status moe_expert_gate_up(const moe_dims *d, const moe_bf16 *hidden, const int32_t *perm,
                                      const int32_t *offsets, const moe_bf16 *w_gate, const moe_bf16 *w_up,
                                      const moe_bf16 *ws_gate, const moe_bf16 *ws_up, void *ws, size_t ws_bytes,
                                      void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;
  if (!ptr_ok(hidden) || !ptr_ok(perm) || !ptr_ok(offsets) || !ptr_ok(w_gate) || !ptr_ok(w_up))
    return MOE_ERR_INVALID_ARG;
  if (d->has_shared && (!ptr_ok(ws_gate) || !ptr_ok(ws_up))) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != MOE_OK) return st;
  return do_gate_up(*d, hidden, perm, offsets, w_gate, w_up, ws_gate, ws_up, ws, (cudaStream_t)stream, true);
}

MOE_API moe_status moe_expert_down(const moe_dims *d, const int32_t *offsets, const moe_bf16 *w_down,
                                   const moe_bf16 *ws_down, moe_bf16 *y_sorted, moe_bf16 *y_shared, void *ws,
                                   size_t ws_bytes, void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;
  if (!ptr_ok(offsets) || !ptr_ok(w_down) || !ptr_ok(y_sorted)) return MOE_ERR_INVALID_ARG;
  if (d->has_shared && (!ptr_ok(ws_down) || !ptr_ok(y_shared))) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != MOE_OK) return st;
  return do_down(*d, offsets, w_down, ws_down, y_sorted, y_shared, ws, (cudaStream_t)stream, true);
}

MOE_API moe_status moe_combine(const moe_dims *d, const moe_bf16 *y_sorted, const moe_bf16 *y_shared,
                               const int32_t *inv_perm, const float *topk_w, moe_bf16 *out, void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;
  if (!ptr_ok(y_sorted) || !ptr_ok(inv_perm) || !ptr_ok(topk_w) || !ptr_ok(out)) return MOE_ERR_INVALID_ARG;
  if (d->has_shared && !ptr_ok(y_shared)) return MOE_ERR_INVALID_ARG;
  return do_combine(*d, y_sorted, y_shared, inv_perm, topk_w, out, (cudaStream_t)stream, true);
}

MOE_API moe_status moe_fused_moe(const moe_dims *d, const moe_bf16 *hidden, const int32_t *topk_idx,
                                 const float *topk_w, const moe_bf16 *w_gate_up, const moe_bf16 *w_down,
                                 const moe_bf16 *ws_gate_up, const moe_bf16 *ws_down, moe_bf16 *out, void *ws,
                                 size_t ws_bytes, void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;
  if (!ptr_ok(hidden) || !ptr_ok(topk_idx) || !ptr_ok(topk_w) || !ptr_ok(w_gate_up) || !ptr_ok(w_down) ||
      !ptr_ok(out))
    return MOE_ERR_INVALID_ARG;
  if (d->has_shared && (!ptr_ok(ws_gate_up) || !ptr_ok(ws_down))) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != MOE_OK) return st;
  return do_fused_moe(*d, hidden, topk_idx, topk_w, w_gate_up, w_down, ws_gate_up, ws_down, out, ws,
                      (cudaStream_t)stream);
}

MOE_API moe_status moe_quantize_fp8_rows(const moe_bf16 *src, int64_t rows, int cols, uint8_t *codes, float *scales,
                                         void *stream) {
  if (rows < 0 || cols <= 0 || cols % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!ptr_ok(src) || !ptr_ok(codes) || scales == nullptr || ((uintptr_t)scales & 3u) != 0) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_rows(reinterpret_cast<const __nv_bfloat16 *>(src), codes, scales, (long long)rows,
                                          cols, (cudaStream_t)stream));
}

MOE_API moe_status moe_expert_ffn_fp8(const moe_dims *d, const moe_bf16 *hidden, const int32_t *perm,
                                      const int32_t *offsets, const moe_fp8_experts *w, moe_bf16 *y_sorted,
                                      moe_bf16 *y_shared, void *ws, size_t ws_bytes, void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;
  if (!ptr_ok(hidden) || !ptr_ok(perm) || !ptr_ok(offsets) || !ptr_ok(y_sorted) || !fp8_ok(*d, w))
    return MOE_ERR_INVALID_ARG;
  if (d->has_shared && !ptr_ok(y_shared)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != MOE_OK) return st;
  return do_expert_phases(*d, 3, hidden, perm, offsets, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                          y_sorted, y_shared, scratch_in(*d, ws), (cudaStream_t)stream, true, 0, w);
}

MOE_API moe_status moe_layer_forward_fp8(const moe_dims *d, const moe_bf16 *hidden, const float *router_w,
                                         const float *expert_bias, const moe_fp8_experts *w, moe_bf16 *out, void *ws,
                                         size_t ws_bytes, void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;
  if (!ptr_ok(hidden) || !ptr_ok(router_w) || !ptr_ok(out) || !fp8_ok(*d, w)) return MOE_ERR_INVALID_ARG;
  if (expert_bias != nullptr && !aligned16(expert_bias)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != MOE_OK) return st;
  const WsLayout L = ws_layout(*d);
  cudaStream_t s = (cudaStream_t)stream;
  int32_t *idx = at<int32_t>(ws, L.topk_idx);
  float *wt = at<float>(ws, L.topk_w);
  int32_t *perm = at<int32_t>(ws, L.perm), *inv = at<int32_t>(ws, L.inv);
  int32_t *offs = at<int32_t>(ws, L.offsets);
  moe_bf16 *y = at<moe_bf16>(ws, L.y_sorted), *z = at<moe_bf16>(ws, L.y_shared);
  if ((st = do_route(*d, hidden, router_w, expert_bias, nullptr, idx, wt, ws, s, true)) != MOE_OK) return st;
  if ((st = do_permute(*d, idx, at<int32_t>(ws, L.counts), offs, perm, inv, ws, s, true)) != MOE_OK) return st;
  if ((st = do_expert_phases(*d, 3, hidden, perm, offs, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, y, z,
                             scratch_in(*d, ws), s, true, 0, w, true)) != MOE_OK)
    return st;
  return do_combine(*d, y, z, inv, wt, out, s, true);
}

// W8A8 needs 128-element K steps: H, I and I_shared multiples of 128.
bool w8a8_shape_ok(const moe_dims &d) {
  return d.H % 128 == 0 && d.I % 128 == 0 && (!d.has_shared || d.I_shared % 128 == 0);
}

MOE_API moe_status moe_expert_ffn_w8a8(const moe_dims *d, const moe_bf16 *hidden, const int32_t *perm,
                                       const int32_t *offsets, const moe_fp8_experts *w, moe_bf16 *y_sorted,
                                       moe_bf16 *y_shared, void *ws, size_t ws_bytes, void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (!w8a8_shape_ok(*d)) return MOE_ERR_UNSUPPORTED;
  if (d->T == 0) return MOE_OK;
  if (!ptr_ok(hidden) || !ptr_ok(perm) || !ptr_ok(offsets) || !ptr_ok(y_sorted) || !fp8_ok(*d, w))
    return MOE_ERR_INVALID_ARG;
  if (d->has_shared && !ptr_ok(y_shared)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const ExpertScratch sc = scratch_in(*d, ws);
  if (launch_quantize_rows(reinterpret_cast<const __nv_bfloat16 *>(hidden), sc.hq, sc.hs, d->T, d->H, s) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return do_expert_phases(*d, 3, hidden, perm, offsets, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                          y_sorted, y_shared, sc, s, true, 0, w, false, true);
}

MOE_API moe_status moe_layer_forward_w8a8(const moe_dims *d, const moe_bf16 *hidden, const float *router_w,
                                          const float *expert_bias, const moe_fp8_experts *w, moe_bf16 *out,
                                          void *ws, size_t ws_bytes, void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (!w8a8_shape_ok(*d)) return MOE_ERR_UNSUPPORTED;
  if (d->T == 0) return MOE_OK;
  if (!ptr_ok(hidden) || !ptr_ok(router_w) || !ptr_ok(out) || !fp8_ok(*d, w)) return MOE_ERR_INVALID_ARG;
  if (expert_bias != nullptr && !aligned16(expert_bias)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != MOE_OK) return st;
  const WsLayout L = ws_layout(*d);
  cudaStream_t s = (cudaStream_t)stream;
  const ExpertScratch sc = scratch_in(*d, ws);
  int32_t *idx = at<int32_t>(ws, L.topk_idx);
  float *wt = at<float>(ws, L.topk_w);
  int32_t *perm = at<int32_t>(ws, L.perm), *inv = at<int32_t>(ws, L.inv);
  int32_t *offs = at<int32_t>(ws, L.offsets);
  moe_bf16 *y = at<moe_bf16>(ws, L.y_sorted), *z = at<moe_bf16>(ws, L.y_shared);
  // the hidden state is quantised first, so that it is complete before the
  // expert kernel's early (routing-independent) tiles read it
  if (launch_quantize_rows(reinterpret_cast<const __nv_bfloat16 *>(hidden), sc.hq, sc.hs, d->T, d->H, s) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if ((st = do_route(*d, hidden, router_w, expert_bias, nullptr, idx, wt, ws, s, true)) != MOE_OK) return st;
  if ((st = do_permute(*d, idx, at<int32_t>(ws, L.counts), offs, perm, inv, ws, s, true)) != MOE_OK) return st;
  if ((st = do_expert_phases(*d, 3, hidden, perm, offs, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, y, z,
                             sc, s, true, 0, w, true, true)) != MOE_OK)
    return st;
  return do_combine(*d, y, z, inv, wt, out, s, true);
}

MOE_API moe_status moe_layer_forward(const moe_dims *d, const moe_bf16 *hidden, const float *router_w,
                                     const float *expert_bias, const moe_bf16 *w_gate, const moe_bf16 *w_up,
                                     const moe_bf16 *w_down, const moe_bf16 *ws_gate, const moe_bf16 *ws_up,
                                     const moe_bf16 *ws_down, moe_bf16 *out, void *ws, size_t ws_bytes,
                                     void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;
  if (!ptr_ok(hidden) || !ptr_ok(router_w) || !ptr_ok(w_gate) || !ptr_ok(w_up) || !ptr_ok(w_down) || !ptr_ok(out))
    return MOE_ERR_INVALID_ARG;
  if (expert_bias != nullptr && !aligned16(expert_bias)) return MOE_ERR_INVALID_ARG;
  if (d->has_shared && (!ptr_ok(ws_gate) || !ptr_ok(ws_up) || !ptr_ok(ws_down))) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != MOE_OK) return st;
  const WsLayout L = ws_layout(*d);
  cudaStream_t s = (cudaStream_t)stream;
  int32_t *idx = at<int32_t>(ws, L.topk_idx);
  float *w = at<float>(ws, L.topk_w);
  int32_t *perm = at<int32_t>(ws, L.perm), *inv = at<int32_t>(ws, L.inv);
  int32_t *offs = at<int32_t>(ws, L.offsets);
  moe_bf16 *y = at<moe_bf16>(ws, L.y_sorted), *z = at<moe_bf16>(ws, L.y_shared);
  if ((st = do_route(*d, hidden, router_w, expert_bias, nullptr, idx, w, ws, s, true)) != MOE_OK) return st;
  if ((st = do_permute(*d, idx, at<int32_t>(ws, L.counts), offs, perm, inv, ws, s, true)) != MOE_OK) return st;
  if ((st = do_expert_ffn(*d, hidden, perm, offs, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, y, z, ws, s,
                          true, true)) != MOE_OK)
    return st;
  return do_combine(*d, y, z, inv, w, out, s, true);
}

// ---------------------------------------------------------------------------
// moe_expert_ffn_noalloc: moe_expert_ffn for callers that cannot allocate
// device memory.  Its scratch (the error word and tile counters, and the bf16
// activations between the gate/up and the down GEMM) lives in the file-scope
// array below instead of a caller-provided workspace, laid out compactly:
// header, then the routed activations [T * top_k, I], then the shared ones [T, I_shared].
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB, held on every device that loads this library
__device__ __align__(256) static unsigned char g_static_scratch[kStaticScratchBytes];

struct NoallocLayout {
  size_t act, act_s, total;
};
NoallocLayout noalloc_layout(const moe_dims &d) {
  NoallocLayout L;
  const size_t S = (size_t)d.T * d.top_k;
  L.act = align256(kWsHeaderBytes);
  L.act_s = align256(L.act + S * (size_t)d.I * 2);
  L.total = L.act_s + (d.has_shared ? (size_t)d.T * d.I_shared * 2 : 0);
  return L;
}

// Device address of the array in the current context (the host-side name is
// not one), looked up with cudaGetSymbolAddress on a context's first call and
// cached under the context's unique id, so that a new context on the same
// device (after cudaDeviceReset, or one the caller made current) gets its own.
constexpr int kScratchCache = 16;
std::mutex g_scratch_mutex;
struct {
  unsigned long long ctx;
  void *ptr;
} g_scratch_cache[kScratchCache] = {};
int g_scratch_next = 0;

void *static_scratch(cudaError_t *err) {
  *err = cudaSuccess;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long ctx = context_id();
  if (ctx != 0)
    for (auto &c : g_scratch_cache)
      if (c.ctx == ctx) return c.ptr;
  void *p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_static_scratch);  // makes the primary context current if none was
  if (*err != cudaSuccess) return nullptr;
  if (ctx == 0) ctx = context_id();
  if (ctx != 0) {
    g_scratch_cache[g_scratch_next] = {ctx, p};
    g_scratch_next = (g_scratch_next + 1) % kScratchCache;
  }
  return p;
}

}  // namespace

MOE_API moe_status moe_expert_ffn_noalloc(const moe_dims *d, const moe_bf16 *hidden, const int32_t *perm,
                                          const int32_t *offsets, const moe_bf16 *w_gate, const moe_bf16 *w_up,
                                          const moe_bf16 *w_down, const moe_bf16 *ws_gate, const moe_bf16 *ws_up,
                                          const moe_bf16 *ws_down, moe_bf16 *y_sorted, moe_bf16 *y_shared,
                                          void *stream) {
  moe_status st = moe_check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;
  if (!ptr_ok(hidden) || !ptr_ok(perm) || !ptr_ok(offsets) || !ptr_ok(w_gate) || !ptr_ok(w_up) || !ptr_ok(w_down) ||
      !ptr_ok(y_sorted))
    return MOE_ERR_INVALID_ARG;
  if (d->has_shared && (!ptr_ok(ws_gate) || !ptr_ok(ws_up) || !ptr_ok(ws_down) || !ptr_ok(y_shared)))
    return MOE_ERR_INVALID_ARG;
  const NoallocLayout L = noalloc_layout(*d);
  if (L.total > kStaticScratchBytes) return MOE_ERR_WORKSPACE;  // beyond the built-in scratch
  cudaError_t e = cudaSuccess;
  void *base = static_scratch(&e);
  if (base == nullptr) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  // the array keeps the previous call's contents: the header (error word and
  // tile-scheduler counters) must start at zero
  if (cudaMemsetAsync(base, 0, kWsHeaderBytes, s) != cudaSuccess) return MOE_ERR_CUDA;
  const ExpertScratch sc = {at<unsigned>(base, 0), at<__nv_bfloat16>(base, L.act), at<__nv_bfloat16>(base, L.act_s)};
  return do_expert_phases(*d, 3, hidden, perm, offsets, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, y_sorted,
                          y_shared, sc, s, true);
}
