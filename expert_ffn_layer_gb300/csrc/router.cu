// Steps a1-a2: router GEMM with the two-BF16 reconstruction of the fp32 router
// weight, then sigmoid+bias (or softmax) scoring, top-k and renormalisation.
//
// "Hy3 Preview inference optimisation case", section 2 (Router GEMM): the fp32
// weight is represented as W_high + W_low / 256; activations stay bf16; two
// BF16 GEMMs accumulate into two accumulators of one kernel and one FFMA in the
// epilogue gives the logits.  hy3 README, Model facts (MoE routing) and the
// HunyuanImage 3.0 post (HunyuanTopKGate easy_topk) give the scoring rules.
//
// Three kernels, chained with programmatic dependent launch:
//   split:  W (fp32) -> W_high, W_low (bf16, [E][H] each) in the workspace, on
//           all SMs (the pages split once offline; here it is one streaming pass).
//   gemm:   a 128-token x Epad-expert tile over one slice of H per CTA; TMA
//           loads x, W_high, W_low; two tcgen05 MMAs per K step into two TMEM
//           accumulators; the epilogue forms acc_lo * (1/256) + acc_hi and
//           writes that slice's partial logits (fp32) to the workspace.
//   topk:   one CTA per token: sums the partial logits of the H slices in a
//           fixed order (deterministic), scores, picks the top-k with warp
//           shuffles, renormalises.
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kSmemLimit = 232448;  // 227 KB opt-in per block
constexpr int kXTileBytes = 128 * 128;  // 128 rows x 64 bf16

// Round fp32 bits to the nearest bf16, ties to even, on the integer pipe (the
// weights are finite): keep the upper 16 bits after adding 0x7FFF plus the
// lowest kept bit.  Returns the rounded value as fp32 bits (low half zero).
__device__ __forceinline__ uint32_t bf16_rne_bits(uint32_t u) {
  return (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
}

__device__ __forceinline__ bool better(float k1, int e1, float k2, int e2) {
  return k1 > k2 || (k1 == k2 && e1 < e2);
}

}  // namespace

// ------------------------------------------------------------------ split
// W_high = bf16_RNE(W), W_low = bf16_RNE((W - W_high) * 256); the difference
// and the scaling by 256 are exact in fp32.  8 weights per thread step.
__global__ void __launch_bounds__(256) router_split_kernel(const float *__restrict__ w, __nv_bfloat16 *w_hi,
                                                           __nv_bfloat16 *w_lo, long long n8) {
  pdl_wait();  // the previous layer may still read the buffers written here
  pdl_launch_dependents();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(w) + 2 * i);
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(w) + 2 * i + 1);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t h[8], l[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      h[j] = bf16_rne_bits(__float_as_uint(v[j]));
      l[j] = bf16_rne_bits(__float_as_uint((v[j] - __uint_as_float(h[j])) * 256.0f));
    }
    reinterpret_cast<uint4 *>(w_hi)[i] =
        make_uint4((h[0] >> 16) | h[1], (h[2] >> 16) | h[3], (h[4] >> 16) | h[5], (h[6] >> 16) | h[7]);
    reinterpret_cast<uint4 *>(w_lo)[i] =
        make_uint4((l[0] >> 16) | l[1], (l[2] >> 16) | l[3], (l[4] >> 16) | l[5], (l[6] >> 16) | l[7]);
  }
}

// ------------------------------------------------------------------ gemm
int router_stages(int Epad) {
  const int stage = kXTileBytes + 2 * Epad * 128;
  int s = (kSmemLimit - 2048) / stage;
  return s > 4 ? 4 : s;
}

size_t router_smem_bytes(int Epad, int stages) { return 1024 + (size_t)stages * (kXTileBytes + 2 * Epad * 128) + 256; }

// Warps: 0 TMA producer (one thread), 1 MMA issuer (one thread) and TMEM owner,
// 2-5 epilogue (TMEM lane quarters 2,3,0,1).
__global__ void __launch_bounds__(kRouterThreads, 1) router_gemm_kernel(const __grid_constant__ RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int Epad = p.Epad;
  const int stage_bytes = kXTileBytes + 2 * Epad * 128;
  const int nst = p.stages;
  uint64_t *bars = (uint64_t *)(smem + nst * stage_bytes);  // full[s], empty[s], done
  uint32_t *tmem_slot = (uint32_t *)(bars + 2 * nst + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = blockIdx.x, m0 = blockIdx.y * 128;
  const int nks = p.kslices_per_cta;
  const int kslice0 = ks * nks;
  uint32_t tmem_cols = 32;
  while (tmem_cols < (uint32_t)(2 * Epad)) tmem_cols <<= 1;
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[nst + s]); };
  const uint32_t done = smem_u32(&bars[2 * nst]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.map_x);
    tma_prefetch_desc(&p.map_hi);
    tma_prefetch_desc(&p.map_lo);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  unsigned *err = p.err;

  pdl_launch_dependents();  // dependents wait for this kernel's completion themselves
  pdl_wait();               // W_high / W_low come from the split kernel

  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < nks && ok; ++i) {
        const int s = i % nst;
        const uint32_t ph = (uint32_t)(i / nst) & 1u;
        ok = mbar_wait(empty(s), ph ^ 1u, err, abort_flag);
        if (!ok) break;
        const uint32_t st = smem_u32(smem + s * stage_bytes);
        mbar_arrive_expect_tx(full(s), (uint32_t)stage_bytes);
        const int k0 = (kslice0 + i) * 64;
        tma_load_2d(st, &p.map_x, full(s), k0, m0);
        tma_load_2d(st + kXTileBytes, &p.map_hi, full(s), k0, 0);
        tma_load_2d(st + kXTileBytes + Epad * 128, &p.map_lo, full(s), k0, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, Epad);
      for (int i = 0; i < nks && ok; ++i) {
        const int s = i % nst;
        const uint32_t ph = (uint32_t)(i / nst) & 1u;
        ok = mbar_wait(full(s), ph, err, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = smem_u32(smem + s * stage_bytes);
        const uint64_t ad = sdesc_sw128(st);
        const uint64_t bh = sdesc_sw128(st + kXTileBytes);
        const uint64_t bl = sdesc_sw128(st + kXTileBytes + Epad * 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          umma_bf16(tmem, ad + 2 * kk, bh + 2 * kk, idesc, acc);
          umma_bf16(tmem + (uint32_t)Epad, ad + 2 * kk, bl + 2 * kk, idesc, acc);
        }
        umma_commit(empty(s));
      }
      umma_commit(done);
    }
  } else {
    // epilogue: partial logits of this H slice = acc_lo * (1/256) + acc_hi
    const int q = warp & 3;
    const int row = 32 * q + lane;
    ok = __all_sync(0xffffffffu, mbar_wait(done, 0, err, abort_flag));
    if (ok) {
      tc_fence_after();
      const uint32_t base = tmem + ((uint32_t)(32 * q) << 16);
      float *dst = p.partial + ((size_t)ks * p.T + m0 + row) * p.E;
      const bool live = m0 + row < p.T;
      for (int c = 0; c < Epad; c += 16) {
        float hi[16], lo[16];
        tmem_ld16(base + (uint32_t)c, hi);
        tmem_ld16(base + (uint32_t)(Epad + c), lo);
        tmem_wait_ld();
        if (live) {
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            if ((p.E & 3) == 0 && c + j + 4 <= p.E) {  // rows are 16-byte aligned only when E % 4 == 0
              const float4 o = make_float4(fmaf(lo[j], 1.0f / 256.0f, hi[j]), fmaf(lo[j + 1], 1.0f / 256.0f, hi[j + 1]),
                                           fmaf(lo[j + 2], 1.0f / 256.0f, hi[j + 2]),
                                           fmaf(lo[j + 3], 1.0f / 256.0f, hi[j + 3]));
              *reinterpret_cast<float4 *>(dst + c + j) = o;
            } else {
              for (int jj = j; jj < j + 4; ++jj)
                if (c + jj < p.E) dst[c + jj] = fmaf(lo[jj], 1.0f / 256.0f, hi[jj]);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// ------------------------------------------------------------------ topk
// Scoring and top-k selection of token t by one warp from its logits lg[0..E).
__device__ __forceinline__ void select_topk(const RouterParams &p, const float *lg, int t, int lane) {
  const int E = p.E, k = p.top_k;
  const int nj = (E + 31) >> 5;
  float v[8], key[8], sc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = (j < nj && lane + 32 * j < E) ? lg[lane + 32 * j] : 0.0f;
  if (p.score_mode == MOE_SCORE_SIGMOID_BIAS) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      const float s = 1.0f / (1.0f + expf(-v[j]));
      const float kk = s + ((p.bias != nullptr && j < nj && e < E) ? p.bias[e] : 0.0f);
      sc[j] = s;
      key[j] = (kk == kk) ? kk : -INFINITY;
    }
  } else {
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < nj && lane + 32 * j < E) mx = fmaxf(mx, v[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float ex[8], sum = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ex[j] = (j < nj && lane + 32 * j < E) ? expf(v[j] - mx) : 0.0f;
      sum += ex[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sc[j] = ex[j] / sum;
      key[j] = (sc[j] == sc[j]) ? sc[j] : -INFINITY;
    }
  }
  uint32_t taken = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (!(j < nj && lane + 32 * j < E)) taken |= 1u << j;
  int my_e = 0;
  float my_s = 0.0f;
  for (int rnd = 0; rnd < k; ++rnd) {
    float bk = -INFINITY, bs = 0.0f;
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      if (!((taken >> j) & 1u) && better(key[j], e, bk, be)) {
        bk = key[j];
        be = e;
        bs = sc[j];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ok2 = __shfl_xor_sync(0xffffffffu, bk, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      const float os = __shfl_xor_sync(0xffffffffu, bs, o);
      if (better(ok2, oe, bk, be)) {
        bk = ok2;
        be = oe;
        bs = os;
      }
    }
    if (be < E && (be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == rnd) {
      my_e = be < E ? be : 0;
      my_s = bs;
    }
  }
  float tot = lane < k ? my_s : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if (lane < k) {
    const float w = p.score_mode == MOE_SCORE_SIGMOID_BIAS ? my_s / tot * p.route_scale : my_s / fmaxf(tot, p.renorm_eps);
    p.topk_idx[(size_t)t * k + lane] = my_e;
    p.topk_w[(size_t)t * k + lane] = w;
  }
}

// TPC tokens per CTA (256 threads).  TPC = 1 (many K slices, small batches):
// thread e sums the KS (<= 32) partial logits of expert e in slice order with
// every load in flight (one round of latency); warp 0 selects.  TPC = 8 (at
// most 4 slices, large batches): the CTA's threads sum the 8 x E logits, then
// warp w selects for the CTA's token w -- all warps select, not one in eight.
template <int TPC>
__global__ void __launch_bounds__(256) router_topk_kernel(const __grid_constant__ RouterParams p, int KS) {
  __shared__ float lg[TPC][256];
  const int t0 = blockIdx.x * TPC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E;
  pdl_launch_dependents();
  pdl_wait();  // the partial logits come from the gemm kernel
  const size_t stride = (size_t)p.T * E;
  // this thread's (token, expert) pairs i = tid + 256 j; every partial of every
  // pair in flight together, then each pair added in slice order
  constexpr int kPairs = (TPC * 256 + 255) / 256;  // pairs per thread (E <= 256)
  constexpr int kMaxKS = TPC == 1 ? 32 : 4;        // slices this form takes
  float part[kPairs][kMaxKS];
#pragma unroll
  for (int j = 0; j < kPairs; ++j) {
    const int i = tid + 256 * j, tok = i / E, e = i - tok * E;
    const bool on = i < TPC * E && t0 + tok < p.T;
    const float *src = p.partial + (size_t)(t0 + tok) * E + e;
#pragma unroll
    for (int s = 0; s < kMaxKS; ++s) part[j][s] = (on && s < KS) ? __ldcg(src + (size_t)s * stride) : 0.0f;
  }
#pragma unroll
  for (int j = 0; j < kPairs; ++j) {
    const int i = tid + 256 * j, tok = i / E, e = i - tok * E;
    if (i < TPC * E && t0 + tok < p.T) {
      float acc = 0.0f;
#pragma unroll
      for (int s = 0; s < kMaxKS; ++s)
        if (s < KS) acc += part[j][s];
      lg[tok][e] = acc;
      if (p.logits_out != nullptr) p.logits_out[(size_t)(t0 + tok) * E + e] = acc;
    }
  }
  __syncthreads();
  if (warp < TPC && t0 + warp < p.T) select_topk(p, lg[warp], t0 + warp, lane);
}

cudaError_t launch_router(const RouterParams &p, const float *router_w, int ksplit, int mtiles, cudaStream_t stream,
                          bool pdl) {
  static thread_local unsigned long long attr_ctx = 0;
  static thread_local int nsm_dev = -1, nsm = 0;
  {
    const cudaError_t e = set_smem_attr_once((const void *)router_gemm_kernel, kSmemLimit, attr_ctx);
    if (e != cudaSuccess) return e;
  }
  int dev = 0;
  cudaGetDevice(&dev);
  if (nsm_dev != dev) {
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    nsm_dev = dev;
  }
  {  // split
    const long long n8 = (long long)p.E * p.H / 8;
    long long blocks = (n8 + 255) / 256;
    if (blocks > 4LL * nsm) blocks = 4LL * nsm;
    const float *w = router_w;
    __nv_bfloat16 *hi = p.w_hi, *lo = p.w_lo;
    long long n = n8;
    void *args[] = {(void *)&w, (void *)&hi, (void *)&lo, (void *)&n};
    cudaError_t e = launch_ex((const void *)router_split_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, pdl, 1,
                              args);
    if (e != cudaSuccess) return e;
  }
  {  // gemm
    void *args[] = {(void *)&p};
    cudaError_t e = launch_ex((const void *)router_gemm_kernel, dim3(ksplit, mtiles, 1), dim3(kRouterThreads, 1, 1),
                              router_smem_bytes(p.Epad, p.stages), stream, true, 1, args);
    if (e != cudaSuccess) return e;
  }
  {  // topk: one token per CTA for small batches, eight for large ones
    int ks = ksplit;
    void *args[] = {(void *)&p, (void *)&ks};
    if (ksplit > 4) return launch_ex((const void *)router_topk_kernel<1>, dim3(p.T), dim3(256), 0, stream, true, 1, args);
    return launch_ex((const void *)router_topk_kernel<8>, dim3((p.T + 7) / 8), dim3(256), 0, stream, true, 1, args);
  }
}

}  // namespace moe
