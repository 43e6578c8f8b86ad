// Step a9: top-k weighted combine back to token order plus the shared branch.
//   out[t] = sum_j w[t, j] * y_sorted[inv[t*k + j]] + y_shared[t]
// "Hy3 Preview inference optimisation case", section 3 (top-k weighted
// aggregation done at the end of the chain); HunyuanImage 3.0 post, Routed
// Experts (outputs viewed as [T, k, H], multiplied by the weights, summed over
// k) and Shared MLP (the shared output is added).
//
// HBM-bound streaming: one thread per 8 hidden values (16-byte vectors), fp32
// accumulation in j order, one bf16 rounding at the end.
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {
constexpr int kThreads = 256;
constexpr int kMaxK = 16;  // top_k limit of the ABI

__device__ __forceinline__ void acc8(float (&a)[8], const uint4 &v, float w) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[2 * i] = fmaf(w, __uint_as_float(u[i] << 16), a[2 * i]);
    a[2 * i + 1] = fmaf(w, __uint_as_float(u[i] & 0xffff0000u), a[2 * i + 1]);
  }
}
}  // namespace

// BATCHED: every slot's loads in flight at once (latency-bound small batches;
// the register cost of top-16 halves residency, which large, bandwidth-bound
// batches need more), else one slot at a time; K8: top-8 exactly, its eight
// rows (and the shared one) in flight together with half that register cost.
// All add in slot order.
template <bool BATCHED, bool K8 = false>
__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int hv = p.H >> 3;
  const long long total = (long long)p.T * hv;
  for (long long idx = (long long)blockIdx.x * kThreads + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * kThreads) {
    const int t = (int)(idx / hv);
    const int c = (int)(idx - (long long)t * hv);
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if constexpr (K8) {
      uint4 v[8];
      float wt[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int pos = min(max(__ldg(p.inv + (size_t)t * 8 + j), 0), p.S - 1);
        wt[j] = __ldg(p.topk_w + (size_t)t * 8 + j);
        v[j] = __ldcs(reinterpret_cast<const uint4 *>(p.y_sorted + (size_t)pos * p.H) + c);
      }
      uint4 z = make_uint4(0u, 0u, 0u, 0u);
      if (p.y_shared != nullptr) z = __ldcs(reinterpret_cast<const uint4 *>(p.y_shared + (size_t)t * p.H) + c);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc8(a, v[j], wt[j]);
      if (p.y_shared != nullptr) acc8(a, z, 1.0f);
    } else if constexpr (!BATCHED) {
      for (int j = 0; j < p.top_k; ++j) {
        const int pos = min(max(__ldg(p.inv + (size_t)t * p.top_k + j), 0), p.S - 1);
        const float w = __ldg(p.topk_w + (size_t)t * p.top_k + j);
        acc8(a, __ldcs(reinterpret_cast<const uint4 *>(p.y_sorted + (size_t)pos * p.H) + c), w);
      }
      if (p.y_shared != nullptr)
        acc8(a, __ldcs(reinterpret_cast<const uint4 *>(p.y_shared + (size_t)t * p.H) + c), 1.0f);
    } else {
      // every slot's index and weight, then every row piece, in flight at once
      // (top_k <= 16); accumulated in slot order
      int pos[kMaxK];
      float wt[kMaxK];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < p.top_k) {
          pos[j] = min(max(__ldg(p.inv + (size_t)t * p.top_k + j), 0), p.S - 1);
          wt[j] = __ldg(p.topk_w + (size_t)t * p.top_k + j);
        }
      }
      uint4 v[kMaxK];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < p.top_k) v[j] = __ldcs(reinterpret_cast<const uint4 *>(p.y_sorted + (size_t)pos[j] * p.H) + c);
      uint4 z = make_uint4(0u, 0u, 0u, 0u);
      if (p.y_shared != nullptr) z = __ldcs(reinterpret_cast<const uint4 *>(p.y_shared + (size_t)t * p.H) + c);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < p.top_k) acc8(a, v[j], wt[j]);
      if (p.y_shared != nullptr) acc8(a, z, 1.0f);
    }
    uint4 o;
    uint32_t *ou = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
      ou[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
    reinterpret_cast<uint4 *>(p.out + (size_t)t * p.H)[c] = o;
  }
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream, bool pdl) {
  static thread_local int nsm = 0, dev_cached = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != dev_cached) {
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    dev_cached = dev;
  }
  const long long total = (long long)p.T * (p.H >> 3);
  long long blocks = (total + kThreads - 1) / kThreads;
  const long long cap = (long long)nsm * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  void *args[] = {(void *)&p};
  const bool batched = total <= (long long)nsm * kThreads;  // one wave of threads
  const void *fn = batched ? (const void *)combine_kernel<true>
                   : p.top_k == 8 ? (const void *)combine_kernel<false, true>
                                  : (const void *)combine_kernel<false>;
  return launch_ex(fn, dim3((unsigned)blocks), dim3(kThreads), 0, stream, pdl, 1, args);
}

}  // namespace moe
