// Steps a5-a8: grouped expert GEMMs over uneven expert segments (plus the
// shared expert as one more segment), on the 5th-generation tensor cores.
//
// "Hy3 Preview inference optimisation case", section 3 (FusedMoE): the gate-up
// GEMM reads the original input through the route index (no explicit gather
// copy); the down GEMM writes compactly per expert.  HunyuanImage 3.0 post:
// SwiGLU experts down(SiLU(gate(x)) * up(x)), stacked expert weights, the
// shared MLP applied to every token.
//
// Orientation ("swap AB"): the weight rows are the M = 128 operand and the
// tokens of one expert chunk are the N operand (N = tokens rounded up to 16,
// at most BN), so an expert with a handful of tokens (decode) costs one
// narrow MMA per K step while its weights stream at full rate, and large
// segments pad to 16 tokens instead of 128.
//
//   gate/up tile: A = [16 gate rows | 16 up rows] x 4 (rows i0..i0+63 of both
//     matrices, interleaved so that gate row i and up row i sit 16 TMEM lanes
//     apart in the same warp), B = token rows gathered with TMA gather4 via
//     perm[p] / k; epilogue: SiLU(gate) * up -> bf16 activation A_act[p][i].
//   down tile:    A = 128 rows of w_down (h0..h0+127), B = A_act rows of the
//     chunk (contiguous); epilogue -> bf16 y_sorted[p][h].
//
// Persistent CTAs (one per SM) walk the tile list in a static stride; the
// tile list (per segment: chunks of <= BN tokens x weight row blocks) is
// derived in every CTA from the expert offsets.  Warp roles: 0 TMA producer,
// 1 tcgen05.mma issuer (one thread), 2-5 epilogue (TMEM -> registers ->
// global).  A STAGES-deep shared-memory ring and two TMEM accumulators let
// loads, MMAs and the epilogue of consecutive tiles overlap.
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kABytes = 128 * 128;  // 128 rows x 64 bf16
constexpr int kMaxSeg = 258;        // E <= 256 routed + 1 shared (+1 sentinel)
constexpr unsigned long long kDrainNs = 20000000ull;

template <int BN>
struct StagesFor {
  static constexpr int value = BN <= 16 ? 12 : BN <= 32 ? 10 : BN <= 64 ? 8 : BN <= 128 ? 6 : 4;
};

template <int BN>
constexpr int tmem_cols_for() {
  return (2 * BN) < 32 ? 32 : 2 * BN;
}

template <int MODE, int BN>
struct Layout {
  static constexpr int kStages = StagesFor<BN>::value;
  static constexpr int kStageBytes = kABytes + BN * 128;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kNumBars = 2 * kStages + 5;  // full, empty, tfull[2], tempty[2], drain
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
  static constexpr int kStartOff = kMiscOff + 16;
  static constexpr int kOffOff = kStartOff + 4 * kMaxSeg;
  static constexpr int kBytes = kOffOff + 4 * kMaxSeg;
  static constexpr size_t kSmem = 1024 + kBytes;
};

struct Tile {
  int seg, rb, row0, ntok, N, nk, shared;
};

// Tokens per chunk for a segment of `cnt` tokens: the fewest chunks of at most
// BN tokens, made as even as possible and rounded up to 16.
template <int BN>
__device__ __forceinline__ int chunk_base(int cnt) {
  const int n0 = (cnt + BN - 1) / BN;
  const int per = (cnt + n0 - 1) / n0;
  return (per + 15) & ~15;
}

template <int MODE>
__device__ __forceinline__ int seg_nrb(const GemmParams &p, bool shared) {
  if (MODE == kGateUp) return (shared ? p.Is : p.I) >> 6;
  return (p.H + 127) >> 7;
}

template <int MODE, int BN>
__device__ __forceinline__ Tile decode_tile(const GemmParams &p, int t, const int *tile_start, const int *seg_off,
                                            int nseg) {
  int lo = 0, hi = nseg;  // tile_start[nseg] = total > t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] <= t) lo = mid;
    else hi = mid;
  }
  Tile tl;
  tl.seg = lo;
  tl.shared = (lo == p.E) ? 1 : 0;
  const int cnt = tl.shared ? p.T : seg_off[lo + 1] - seg_off[lo];
  const int nrb = seg_nrb<MODE>(p, tl.shared);
  const int local = t - tile_start[lo];
  const int ch = local / nrb;
  tl.rb = local - ch * nrb;
  const int base = chunk_base<BN>(cnt);
  const int pin = ch * base;
  tl.ntok = min(base, cnt - pin);
  tl.row0 = (tl.shared ? 0 : seg_off[lo]) + pin;
  tl.N = (tl.ntok + 15) & ~15;
  tl.nk = MODE == kGateUp ? (p.H >> 6) : ((tl.shared ? p.Is : p.I) >> 6);
  return tl;
}

__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kDrainNs) return false;
  return true;
}

}  // namespace

template <int MODE, int BN>
__global__ void __launch_bounds__(kGemmThreads, 1) expert_gemm_kernel(const __grid_constant__ GemmParams p) {
  using L = Layout<MODE, BN>;
  constexpr int STAGES = L::kStages;
  constexpr uint32_t kTmemCols = tmem_cols_for<BN>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = (uint64_t *)(smem + L::kBarOff);
  uint32_t *tmem_slot = (uint32_t *)(smem + L::kMiscOff);
  volatile int *abort_flag = (volatile int *)(smem + L::kMiscOff + 4);
  int *tile_start = (int *)(smem + L::kStartOff);
  int *seg_off = (int *)(smem + L::kOffOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[STAGES + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + 2 + a]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * STAGES + 4]);
  auto a_smem = [&](int s) { return smem_u32(smem + s * L::kStageBytes); };
  auto b_smem = [&](int s) { return smem_u32(smem + s * L::kStageBytes + kABytes); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.map_a0);
    tma_prefetch_desc(&p.map_b);
    if (MODE == kGateUp) tma_prefetch_desc(&p.map_a1);
    if (p.has_shared) tma_prefetch_desc(&p.map_s0);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_wait();  // perm / offsets / activations come from the previous kernel
  pdl_launch_dependents();

  // ---------------- tile list from the expert offsets (warp 2)
  const int nseg = p.E + (p.has_shared ? 1 : 0);
  if (warp == 2) {
    for (int i = lane; i <= p.E; i += 32) seg_off[i] = __ldg(p.offsets + i);
    __syncwarp();
    bool good = true;
    for (int i = lane; i <= p.E; i += 32) {
      if (i == 0) good = good && seg_off[0] == 0;
      else good = good && seg_off[i] >= seg_off[i - 1];
      if (i == p.E) good = good && seg_off[i] == p.S;
    }
    good = __all_sync(0xffffffffu, good);
    if (!good && blockIdx.x == 0 && lane == 0 && p.err != nullptr) atomicOr(p.err, MOE_DEVERR_OFFSETS);
    const int per = (nseg + 31) / 32;
    const int s0 = lane * per;
    int local = 0;
    for (int s = s0; s < min(nseg, s0 + per); ++s) {
      const bool sh = (s == p.E);
      const int cnt = sh ? p.T : seg_off[s + 1] - seg_off[s];
      const int chunks = cnt > 0 ? (cnt + chunk_base<BN>(cnt) - 1) / chunk_base<BN>(cnt) : 0;
      local += good ? chunks * seg_nrb<MODE>(p, sh) : 0;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int run = incl - local;
    for (int s = s0; s < min(nseg, s0 + per); ++s) {
      tile_start[s] = run;
      const bool sh = (s == p.E);
      const int cnt = sh ? p.T : seg_off[s + 1] - seg_off[s];
      const int chunks = cnt > 0 ? (cnt + chunk_base<BN>(cnt) - 1) / chunk_base<BN>(cnt) : 0;
      run += good ? chunks * seg_nrb<MODE>(p, sh) : 0;
    }
    if (lane == 31) tile_start[nseg] = incl;
  }
  __syncthreads();
  const int total = tile_start[nseg];
  unsigned *err = p.err;
  bool ok = true;

  if (warp == 0) {
    // ================= TMA producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    int st = 0;
    uint32_t ph = 0;
    uint32_t issued = 0, issued_par = 0;  // per stage: has a load been issued, and its phase parity
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = decode_tile<MODE, BN>(p, t, tile_start, seg_off, nseg);
      int rows[8];
      bool bad = false;
      if (MODE == kGateUp) {
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
          const int g = lane + 32 * gi;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = 4 * g + q;
            const int rr = r < tl.ntok ? r : 0;
            int tok = 0;
            if (g * 4 < tl.N) {
              if (tl.shared) {
                tok = tl.row0 + rr;
              } else {
                const int slot = __ldg(p.perm + tl.row0 + rr);
                tok = slot / p.top_k;
                if (slot < 0 || tok >= p.T) {
                  bad = true;
                  tok = 0;
                }
              }
            }
            rows[gi * 4 + q] = tok;
          }
        }
        if (bad && err != nullptr) atomicOr(err, MOE_DEVERR_INDEX);
      }
      const uint32_t tx = (uint32_t)(kABytes + tl.N * 128);
      for (int kb = 0; kb < tl.nk; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(empty_bar(st), ph ^ 1u, err, abort_flag));
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(full_bar(st), tx);
          issued |= 1u << st;
          issued_par = (issued_par & ~(1u << st)) | (ph << st);
        }
        __syncwarp();
        const int k0 = kb * 64;
        if (lane == 0) {
          if (MODE == kGateUp) {
            const int i0 = tl.rb * 64;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t dg = a_smem(st) + (uint32_t)(32 * q) * 128;
              const uint32_t du = dg + 16 * 128;
              if (tl.shared) {
                tma_load_2d_hint(dg, &p.map_s0, full_bar(st), k0, i0 + 16 * q, pol_w);
                tma_load_2d_hint(du, &p.map_s1, full_bar(st), k0, i0 + 16 * q, pol_w);
              } else {
                tma_load_3d_hint(dg, &p.map_a0, full_bar(st), k0, i0 + 16 * q, tl.seg, pol_w);
                tma_load_3d_hint(du, &p.map_a1, full_bar(st), k0, i0 + 16 * q, tl.seg, pol_w);
              }
            }
          } else {
            const int h0 = tl.rb * 128;
            if (tl.shared) tma_load_2d_hint(a_smem(st), &p.map_s0, full_bar(st), k0, h0, pol_w);
            else tma_load_3d_hint(a_smem(st), &p.map_a0, full_bar(st), k0, h0, tl.seg, pol_w);
          }
        }
        if (MODE == kGateUp) {
#pragma unroll
          for (int gi = 0; gi < 2; ++gi) {
            const int g = lane + 32 * gi;
            if (g * 4 < tl.N)
              tma_gather4(b_smem(st) + (uint32_t)g * 512, &p.map_b, full_bar(st), k0, rows[gi * 4 + 0],
                          rows[gi * 4 + 1], rows[gi * 4 + 2], rows[gi * 4 + 3], pol_x);
          }
        } else {
          if (lane * 16 < tl.N) {
            const CUtensorMap *mb = tl.shared ? &p.map_bs : &p.map_b;
            tma_load_2d_hint(b_smem(st) + (uint32_t)lane * 2048, mb, full_bar(st), k0, tl.row0 + 16 * lane, pol_x);
          }
        }
        if (++st == STAGES) {
          st = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      // let every load this CTA issued land before the block exits
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) mbar_wait_drain(full_bar(s), (issued_par >> s) & 1u);
    }
  } else if (warp == 1) {
    // ================= MMA issuer
    if (lane == 0) {
      int st = 0, it = 0;
      uint32_t ph = 0;
      bool any = false;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const Tile tl = decode_tile<MODE, BN>(p, t, tile_start, seg_off, nseg);
        const int acc = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        ok = mbar_wait(tempty_bar(acc), aph ^ 1u, err, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * BN);
        const uint32_t idesc = idesc_bf16(128, tl.N);
        for (int kb = 0; kb < tl.nk; ++kb) {
          ok = mbar_wait(full_bar(st), ph, err, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(a_smem(st));
          const uint64_t bd = sdesc_sw128(b_smem(st));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          any = true;
          umma_commit(empty_bar(st));
          if (++st == STAGES) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
      }
      if (!ok && any) {
        umma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0);
      }
    }
  } else {
    // ================= epilogue (warps 2..5 -> TMEM lane quarters 2,3,0,1)
    const int q = warp & 3;
    int it = 0;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
      const Tile tl = decode_tile<MODE, BN>(p, t, tile_start, seg_off, nseg);
      const int acc = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), aph, err, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
      if (MODE == kGateUp) {
        const int ld = tl.shared ? p.Is : p.I;
        __nv_bfloat16 *out = tl.shared ? p.out_s : p.out;
        const int i = tl.rb * 64 + 16 * q + (lane & 15);
        const bool upper = lane >= 16;
        for (int c = 0; c < tl.N; c += 16) {
          float v[16];
          tmem_ld16(taddr + (uint32_t)c, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float send = upper ? v[j] : v[j + 1];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
            const float g = upper ? recv : v[j];
            const float u = upper ? v[j + 1] : recv;
            const int col = c + j + (upper ? 1 : 0);
            const float a = g / (1.0f + __expf(-g)) * u;
            if (col < tl.ntok) out[(size_t)(tl.row0 + col) * ld + i] = __float2bfloat16_rn(a);
          }
        }
      } else {
        __nv_bfloat16 *out = tl.shared ? p.out_s : p.out;
        const int h = tl.rb * 128 + 32 * q + lane;
        for (int c = 0; c < tl.N; c += 16) {
          float v[16];
          tmem_ld16(taddr + (uint32_t)c, v);
          tmem_wait_ld();
          if (h < p.H) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c + j < tl.ntok) out[(size_t)(tl.row0 + c + j) * p.H + h] = __float2bfloat16_rn(v[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
    }
  }

  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int gemm_tile_n(int T) {
  if (T <= 16) return 16;
  if (T <= 32) return 32;
  if (T <= 64) return 64;
  if (T <= 128) return 128;
  return 256;
}

namespace {
template <int MODE, int BN>
cudaError_t launch_one(const GemmParams &p, int num_ctas, cudaStream_t stream, bool pdl) {
  using L = Layout<MODE, BN>;
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(expert_gemm_kernel<MODE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::kSmem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  void *args[] = {(void *)&p};
  return launch_ex((const void *)expert_gemm_kernel<MODE, BN>, dim3(num_ctas), dim3(kGemmThreads), L::kSmem, stream,
                   pdl, 1, args);
}

template <int MODE>
cudaError_t launch_mode(const GemmParams &p, int bn, int num_ctas, cudaStream_t stream, bool pdl) {
  switch (bn) {
    case 16: return launch_one<MODE, 16>(p, num_ctas, stream, pdl);
    case 32: return launch_one<MODE, 32>(p, num_ctas, stream, pdl);
    case 64: return launch_one<MODE, 64>(p, num_ctas, stream, pdl);
    case 128: return launch_one<MODE, 128>(p, num_ctas, stream, pdl);
    case 256: return launch_one<MODE, 256>(p, num_ctas, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_expert_gemm(const GemmParams &p, GemmMode mode, int bn, int num_ctas, cudaStream_t stream,
                               bool pdl) {
  return mode == kGateUp ? launch_mode<kGateUp>(p, bn, num_ctas, stream, pdl)
                         : launch_mode<kDown>(p, bn, num_ctas, stream, pdl);
}

}  // namespace moe
