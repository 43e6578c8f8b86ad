// Steps a1-a2: router GEMM with the two-BF16 reconstruction of the fp32 router
// weight, then sigmoid+bias (or softmax) scoring, top-k and renormalisation.
//
// "Hy3 Preview inference optimisation case", section 2 (Router GEMM): the fp32
// weight is represented as W_high + W_low / 256; activations stay bf16; two
// BF16 GEMMs accumulate into two accumulators of one kernel and one FFMA in the
// epilogue gives the logits.  hy3 README, Model facts (MoE routing) and the
// HunyuanImage 3.0 post (HunyuanTopKGate easy_topk) give the scoring rules.
//
// One CTA computes a 128-token x Epad-expert tile over a slice of H; the
// KS CTAs of a thread-block cluster split H and reduce their partial logits
// through distributed shared memory in a fixed order (deterministic), then
// one warp per token row does the top-k with warp shuffles.
//
// Warp roles: 0-3 convert fp32 W tiles into W_high / W_low (in place, in
// shared memory) and later run the epilogue; 4 issues tcgen05.mma; 5 issues TMA.
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kSmemLimit = 232448;  // 227 KB opt-in per block
constexpr int kXTileBytes = 128 * 128;  // 128 rows x 64 bf16

__device__ __forceinline__ uint64_t sdesc_noswizzle(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version; layout type 0 = no swizzle
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// Split 8 fp32 into 8 W_high and 8 W_low bf16 (each a 16-byte row of a core matrix).
__device__ __forceinline__ void split8(const float4 &a, const float4 &b, uint4 &hi, uint4 &lo) {
  float w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  __nv_bfloat16 h[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = __float2bfloat16_rn(w[i]);
    const float r = w[i] - __bfloat162float(h[i]);  // exact in fp32
    l[i] = __float2bfloat16_rn(r * 256.0f);          // exact scaling, one rounding
  }
  hi = make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]), pack_bf16x2(h[6], h[7]));
  lo = make_uint4(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]), pack_bf16x2(l[4], l[5]), pack_bf16x2(l[6], l[7]));
}

__device__ __forceinline__ bool better(float k1, int e1, float k2, int e2) {
  return k1 > k2 || (k1 == k2 && e1 < e2);
}

}  // namespace

int router_stages(int Epad) {
  const int stage = kXTileBytes + Epad * 256;
  int s = (kSmemLimit - 2048) / stage;
  return s > 3 ? 3 : s;
}

size_t router_smem_bytes(int Epad, int stages) {
  return 1024 + (size_t)stages * (kXTileBytes + Epad * 256) + 512;
}

__global__ void __launch_bounds__(kRouterThreads, 1) router_kernel(const __grid_constant__ RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int Epad = p.Epad;
  const int stage_bytes = kXTileBytes + Epad * 256;
  const int nst = p.stages;
  uint64_t *bars = (uint64_t *)(smem + nst * stage_bytes);
  // loaded[s], converted[s], empty[s], done
  uint32_t *tmem_slot = (uint32_t *)(bars + 3 * nst + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t KS = gridDim.x;  // the cluster spans x
  const int m0 = blockIdx.y * 128;
  const int nks = p.kslices_per_cta;
  const int kslice0 = (int)rank * nks;
  uint32_t tmem_cols = 32;
  while (tmem_cols < (uint32_t)(2 * Epad)) tmem_cols <<= 1;

  auto loaded = [&](int s) { return smem_u32(&bars[s]); };
  auto converted = [&](int s) { return smem_u32(&bars[nst + s]); };
  auto emptyb = [&](int s) { return smem_u32(&bars[2 * nst + s]); };
  const uint32_t done = smem_u32(&bars[3 * nst]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(loaded(s), 1);
      mbar_init(converted(s), 128);
      mbar_init(emptyb(s), 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5 && lane == 0) {
    tma_prefetch_desc(&p.map_x);
    tma_prefetch_desc(&p.map_w);
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  unsigned *err = p.err;

  pdl_wait();  // hidden may come from the previous kernel of a chain
  pdl_launch_dependents();

  bool ok = true;
  if (warp == 5) {
    // ---------------- TMA producer
    if (lane == 0) {
      for (int i = 0; i < nks && ok; ++i) {
        const int s = i % nst;
        const uint32_t ph = (uint32_t)(i / nst) & 1u;
        ok = mbar_wait(emptyb(s), ph ^ 1u, err, abort_flag);
        if (!ok) break;
        uint8_t *st = smem + s * stage_bytes;
        mbar_arrive_expect_tx(loaded(s), (uint32_t)stage_bytes);
        const int k0 = (kslice0 + i) * 64;
        tma_load_2d(smem_u32(st), &p.map_x, loaded(s), k0, m0);
        tma_load_2d(smem_u32(st + kXTileBytes), &p.map_w, loaded(s), k0, 0);
      }
    }
  } else if (warp == 4) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, Epad);
      for (int i = 0; i < nks && ok; ++i) {
        const int s = i % nst;
        const uint32_t ph = (uint32_t)(i / nst) & 1u;
        ok = mbar_wait(converted(s), ph, err, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t xs = smem_u32(smem + s * stage_bytes);
        const uint32_t ws = xs + kXTileBytes;
        const uint64_t adesc = sdesc_sw128(xs);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // W_high core matrices at group*2048 + kgroup*128; W_low at +1024
          const uint64_t bh = sdesc_noswizzle(ws + kk * 256, 128, 2048);
          const uint64_t bl = sdesc_noswizzle(ws + 1024 + kk * 256, 128, 2048);
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          umma_bf16(tmem, adesc + 2 * kk, bh, idesc, acc);
          umma_bf16(tmem + (uint32_t)Epad, adesc + 2 * kk, bl, idesc, acc);
        }
        umma_commit(emptyb(s));
      }
      umma_commit(done);
    }
  } else {
    // ---------------- converters: fp32 rows -> W_high / W_low core matrices, in place
    const int r = lane & 7, q = lane >> 3;  // row within an 8-row group, 16-float quarter
    for (int i = 0; i < nks && ok; ++i) {
      const int s = i % nst;
      const uint32_t ph = (uint32_t)(i / nst) & 1u;
      ok = __all_sync(0xffffffffu, mbar_wait(loaded(s), ph, err, abort_flag));
      if (!ok) break;
      uint8_t *wst = smem + s * stage_bytes + kXTileBytes;
      for (int g = warp; g < Epad / 8; g += 4) {
        uint8_t *region = wst + g * 2048;  // rows 8g..8g+7, 256 B each (64 fp32)
        // a[j] holds 16-byte chunk (j + r) & 3 of this lane's quarter: the rotation
        // spreads the 8 rows of a phase over 4 bank groups.
        float4 a[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = 4 * q + ((j + r) & 3);
          a[j] = *reinterpret_cast<const float4 *>(region + r * 256 + c * 16);
        }
        const int rot = r & 3;  // v[m] = a[(m - rot) & 3], with static indices only
        float4 v[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          v[m] = a[m];
          if (rot == 1) v[m] = a[(m + 3) & 3];
          if (rot == 2) v[m] = a[(m + 2) & 3];
          if (rot == 3) v[m] = a[(m + 1) & 3];
        }
        uint4 hi0, lo0, hi1, lo1;
        split8(v[0], v[1], hi0, lo0);  // k = 16q .. 16q+7  -> k-group 2q
        split8(v[2], v[3], hi1, lo1);  // k = 16q+8 .. 16q+15 -> k-group 2q+1
        __syncwarp();
        *reinterpret_cast<uint4 *>(region + (2 * q) * 128 + r * 16) = hi0;
        *reinterpret_cast<uint4 *>(region + (2 * q + 1) * 128 + r * 16) = hi1;
        *reinterpret_cast<uint4 *>(region + 1024 + (2 * q) * 128 + r * 16) = lo0;
        *reinterpret_cast<uint4 *>(region + 1024 + (2 * q + 1) * 128 + r * 16) = lo1;
        __syncwarp();
      }
      fence_proxy_async_smem();
      mbar_arrive(converted(s));
    }
  }

  // ---------------- epilogue: logits = acc_lo * (1/256) + acc_hi  ->  smem tile [128][Epad+1]
  float *tile = reinterpret_cast<float *>(smem);
  const int ld = Epad + 1;
  const int rows_valid = min(128, p.T - m0);
  __syncwarp();
  if (warp < 4) {
    ok = __all_sync(0xffffffffu, ok && mbar_wait(done, 0, err, abort_flag));
    if (ok) {
      tc_fence_after();
      const int row = warp * 32 + lane;
      const uint32_t base = tmem + ((uint32_t)(warp * 32) << 16);
      for (int c = 0; c < Epad; c += 16) {
        float hi[16], lo[16];
        tmem_ld16(base + (uint32_t)c, hi);
        tmem_ld16(base + (uint32_t)(Epad + c), lo);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) tile[row * ld + c + j] = fmaf(lo[j], 1.0f / 256.0f, hi[j]);
      }
    }
  }
  tc_fence_before();
  cluster_sync();

  // ---------------- cluster reduce (fixed order over the KS slices) + top-k, one warp per row
  if (!*abort_flag) {
    const uint32_t tile_s = smem_u32(tile);
    const int E = p.E, k = p.top_k;
    const int nj = (E + 31) >> 5;
    for (int i = (int)rank + (int)KS * warp; i < rows_valid; i += (int)KS * (kRouterThreads / 32)) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = 0.0f;
        const int e = lane + 32 * j;
        if (j < nj && e < E) {
          const uint32_t a = tile_s + (uint32_t)((i * ld + e) * 4);
          float acc = 0.0f;
          for (uint32_t rr = 0; rr < KS; ++rr) acc += ld_cluster_f32(map_cluster(a, rr));
          v[j] = acc;
          if (p.logits_out != nullptr) p.logits_out[(size_t)(m0 + i) * E + e] = acc;
        }
      }
      // scores and keys
      float key[8], sc[8];
      if (p.score_mode == MOE_SCORE_SIGMOID_BIAS) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int e = lane + 32 * j;
          const float s = 1.0f / (1.0f + expf(-v[j]));
          float kk = s + ((p.bias != nullptr && j < nj && e < E) ? p.bias[e] : 0.0f);
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
        const float w = p.score_mode == MOE_SCORE_SIGMOID_BIAS ? my_s / tot * p.route_scale
                                                               : my_s / fmaxf(tot, p.renorm_eps);
        p.topk_idx[(size_t)(m0 + i) * k + lane] = my_e;
        p.topk_w[(size_t)(m0 + i) * k + lane] = w;
      }
    }
  }
  cluster_sync();  // remote CTAs may still read this CTA's tile until here
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

cudaError_t launch_router(const RouterParams &p, int ksplit, int mtiles, cudaStream_t stream, bool pdl) {
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  void *args[] = {(void *)&p};
  return launch_ex((const void *)router_kernel, dim3(ksplit, mtiles, 1), dim3(kRouterThreads, 1, 1),
                   router_smem_bytes(p.Epad, p.stages), stream, pdl, ksplit, args);
}

}  // namespace moe
