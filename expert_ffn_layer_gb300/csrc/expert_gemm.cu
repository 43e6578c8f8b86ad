// Steps a5-a8: grouped expert GEMMs over uneven expert segments (plus the
// shared expert as one more segment), on the 5th-generation tensor cores.
//
// "Hy3 Preview inference optimisation case", section 3 (FusedMoE): the gate-up
// GEMM reads the original input through the route index (no explicit gather
// copy); the down GEMM writes compactly per expert.  HunyuanImage 3.0 post:
// SwiGLU experts down(SiLU(gate(x)) * up(x)), stacked expert weights, the
// shared MLP applied to every token.
//
// Orientation: weight rows are the M = 128 operand of every MMA and the tokens
// of one expert chunk are the N operand (N = tokens rounded up to 16, at most
// BN <= 256).  A tile is 256 weight rows x N tokens: two MMAs per K step share
// one token tile and accumulate into two TMEM accumulators,
//   gate/up: D0 = gate rows i0..i0+127, D1 = up rows i0..i0+127, so gate row i
//            and up row i land in the same TMEM lane and one thread forms
//            SiLU(gate) * up -> bf16 activation A_act[p][i];
//   down:    D0 = w_down rows h0..h0+127, D1 = rows h0+128..h0+255 -> y[p][h].
// Sharing the token tile between 256 weight rows halves the token re-reads
// from L2 compared with one 128-row MMA per tile.
//
// Operand loads per 64-wide K step: the two 128-row weight boxes by TMA
// (128-byte swizzle); the token rows of gate/up through the route index
// (token = perm[p] / k) by cp.async from 128 producer threads straight from
// `hidden`, written in the same swizzled layout (TMA's row-gather moves 4 rows
// per instruction and tops out far below the rate these tiles need); the
// activation rows of down, which are contiguous, by at most four TMA boxes.
//
// Persistent CTAs (one per SM) walk the tile list in a static stride; the
// tile list (per segment: weight row blocks x chunks of <= BN tokens, chunks
// innermost so chunks of one row block reuse its weights in L2) is derived in
// every CTA from the expert offsets.  Warp roles: 0-3 producers, 4 MMA issuer
// (one thread) and TMEM owner, 5-8 epilogue.  A STAGES-deep shared-memory
// ring overlaps loads and MMAs; for BN <= 128 two TMEM accumulator pairs also
// overlap one tile's epilogue with the next tile's MMAs (BN = 256 fills TMEM
// with one pair).
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kABytes = 2 * 128 * 128;  // two 128-row x 64-bf16 weight boxes
constexpr int kMaxSeg = 258;            // E <= 256 routed + 1 shared (+1 sentinel)
constexpr int kProducers = 128;         // warps 0-3
constexpr int kMmaWarp = 4;
constexpr unsigned long long kDrainNs = 20000000ull;

template <int BN>
struct StagesFor {
  static constexpr int value = BN <= 32 ? 6 : BN <= 64 ? 5 : BN <= 128 ? 4 : 3;
};

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
  // accumulator pairs of 2 x BN columns: two (MMA of the next tile overlaps the
  // epilogue of this one) while they fit in the 512 TMEM columns, else one
  static constexpr int kAccBufs = 4 * BN <= 512 ? 2 : 1;
  static constexpr uint32_t kTmemCols = kAccBufs * 2 * BN;
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kTmemCols >= 32 && kTmemCols <= 512, "TMEM budget");
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
template <int BN>
__device__ __forceinline__ int chunk_count(int cnt) {
  if (cnt <= 0) return 0;
  const int b = chunk_base<BN>(cnt);
  return (cnt + b - 1) / b;
}

// Weight row blocks of a segment: 128 gate/up pairs, or 256 rows of w_down.
template <int MODE>
__device__ __forceinline__ int seg_nrb(const GemmParams &p, bool shared) {
  if (MODE == kGateUp) return ((shared ? p.Is : p.I) + 127) >> 7;
  return (p.H + 255) >> 8;
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
  const int nch = chunk_count<BN>(cnt);
  const int local = t - tile_start[lo];
  tl.rb = local / nch;
  const int ch = local - tl.rb * nch;
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

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed (the
// arrival is one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

}  // namespace

template <int MODE, int BN>
__global__ void __launch_bounds__(kGemmThreads, 1) expert_gemm_kernel(const __grid_constant__ GemmParams p) {
  using L = Layout<MODE, BN>;
  constexpr int STAGES = L::kStages;
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
      // gate/up: 128 cp.async arrivals + the TMA expect_tx arrival; down: TMA only
      mbar_init(full_bar(s), MODE == kGateUp ? kProducers + 1 : 1);
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
    if (MODE == kGateUp) tma_prefetch_desc(&p.map_a1);
    if (p.has_shared) tma_prefetch_desc(&p.map_s0);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_wait();  // perm / offsets / activations come from the previous kernel
  pdl_launch_dependents();

  // ---------------- tile list from the expert offsets (one warp)
  const int nseg = p.E + (p.has_shared ? 1 : 0);
  if (warp == kMmaWarp) {
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
      local += good ? chunk_count<BN>(cnt) * seg_nrb<MODE>(p, sh) : 0;
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
      run += good ? chunk_count<BN>(cnt) * seg_nrb<MODE>(p, sh) : 0;
    }
    if (lane == 31) tile_start[nseg] = incl;
  }
  __syncthreads();
  const int total = tile_start[nseg];
  unsigned *err = p.err;
  bool ok = true;

  if (warp < 4) {
    // ================= producers
    const bool tma_thread = threadIdx.x == 0;
    const uint64_t pol_w = policy_evict_first();
    int st = 0;
    uint32_t ph = 0;
    uint32_t issued = 0, issued_par = 0;  // per stage: TMA issued, and its phase parity (thread 0)
    if (MODE == kGateUp || warp == 0) {
      const int tid = threadIdx.x;          // 0..127
      const int c8 = tid & 7, rbase = tid >> 3;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = decode_tile<MODE, BN>(p, t, tile_start, seg_off, nseg);
        // token rows of this thread (gate/up): rows rbase + 16 j of the chunk
        const __nv_bfloat16 *src[BN / 16];
        if (MODE == kGateUp) {
          bool bad = false;
#pragma unroll
          for (int j = 0; j < BN / 16; ++j) {
            const int r = rbase + 16 * j;
            const int rr = r < tl.ntok ? r : 0;
            int tok = 0;
            if (r < tl.N) {
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
            src[j] = p.hidden + (size_t)tok * p.H + c8 * 8;
          }
          if (bad && err != nullptr) atomicOr(err, MOE_DEVERR_INDEX);
        }
        const int i0 = tl.rb * (MODE == kGateUp ? 128 : 256);
        for (int kb = 0; kb < tl.nk; ++kb) {
          ok = __all_sync(0xffffffffu, mbar_wait(empty_bar(st), ph ^ 1u, err, abort_flag));
          if (!ok) break;
          const int k0 = kb * 64;
          if (tma_thread) {
            const uint32_t tx = MODE == kGateUp ? (uint32_t)kABytes : (uint32_t)(kABytes + tl.N * 128);
            mbar_arrive_expect_tx(full_bar(st), tx);
            issued |= 1u << st;
            issued_par = (issued_par & ~(1u << st)) | (ph << st);
            const uint32_t a0 = a_smem(st), a1 = a0 + 16384;
            if (MODE == kGateUp) {
              if (tl.shared) {
                tma_load_2d_hint(a0, &p.map_s0, full_bar(st), k0, i0, pol_w);
                tma_load_2d_hint(a1, &p.map_s1, full_bar(st), k0, i0, pol_w);
              } else {
                tma_load_3d_hint(a0, &p.map_a0, full_bar(st), k0, i0, tl.seg, pol_w);
                tma_load_3d_hint(a1, &p.map_a1, full_bar(st), k0, i0, tl.seg, pol_w);
              }
            } else {
              if (tl.shared) {
                tma_load_2d_hint(a0, &p.map_s0, full_bar(st), k0, i0, pol_w);
                tma_load_2d_hint(a1, &p.map_s0, full_bar(st), k0, i0 + 128, pol_w);
              } else {
                tma_load_3d_hint(a0, &p.map_a0, full_bar(st), k0, i0, tl.seg, pol_w);
                tma_load_3d_hint(a1, &p.map_a0, full_bar(st), k0, i0 + 128, tl.seg, pol_w);
              }
              // activation rows row0 .. row0 + N (contiguous, N a multiple of 16 and
              // <= 256): boxes of 128 rows while they fit, then one each of 64/32/16
              const CUtensorMap *mb = tl.shared ? p.map_bs : p.map_b;
              int off = 0;
              while (tl.N - off >= 128) {
                tma_load_2d(b_smem(st) + (uint32_t)off * 128, &mb[3], full_bar(st), k0, tl.row0 + off);
                off += 128;
              }
#pragma unroll
              for (int bi = 2; bi >= 0; --bi) {
                const int h = 16 << bi;
                if (tl.N - off >= h) {
                  tma_load_2d(b_smem(st) + (uint32_t)off * 128, &mb[bi], full_bar(st), k0, tl.row0 + off);
                  off += h;
                }
              }
            }
          }
          if (MODE == kGateUp) {
            const uint32_t bs = b_smem(st);
#pragma unroll
            for (int j = 0; j < BN / 16; ++j) {
              const int r = rbase + 16 * j;
              if (r < tl.N) cp_async_16(bs + r * 128 + ((c8 ^ (r & 7)) << 4), src[j] + k0);
            }
            cp_async_arrive_noinc(full_bar(st));
          }
          if (++st == STAGES) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        if (MODE == kGateUp) cp_async_wait_all();
        if (tma_thread)
          for (int s = 0; s < STAGES; ++s)
            if ((issued >> s) & 1u) mbar_wait_drain(full_bar(s), (issued_par >> s) & 1u);
      }
    }
  } else if (warp == kMmaWarp) {
    // ================= MMA issuer
    if (lane == 0) {
      int st = 0, it = 0;
      uint32_t ph = 0;
      bool any = false;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const Tile tl = decode_tile<MODE, BN>(p, t, tile_start, seg_off, nseg);
        const int acc = it % L::kAccBufs;
        const uint32_t aph = (uint32_t)(it / L::kAccBufs) & 1u;
        ok = mbar_wait(tempty_bar(acc), aph ^ 1u, err, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)(acc * 2 * BN);
        const uint32_t d1 = d0 + (uint32_t)BN;
        const uint32_t idesc = idesc_bf16(128, tl.N);
        for (int kb = 0; kb < tl.nk; ++kb) {
          ok = mbar_wait(full_bar(st), ph, err, abort_flag);
          if (!ok) break;
          if (MODE == kGateUp) fence_proxy_async_smem();  // token rows were written by cp.async
          tc_fence_after();
          const uint64_t a0 = sdesc_sw128(a_smem(st));
          const uint64_t a1 = sdesc_sw128(a_smem(st) + 16384);
          const uint64_t bd = sdesc_sw128(b_smem(st));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            umma_bf16(d0, a0 + 2 * kk, bd + 2 * kk, idesc, accum);
            umma_bf16(d1, a1 + 2 * kk, bd + 2 * kk, idesc, accum);
          }
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
    // ================= epilogue (warps 5..8 -> TMEM lane quarters 1,2,3,0)
    const int q = warp & 3;
    const int r = 32 * q + lane;  // weight row within the 128-row half
    int it = 0;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
      const Tile tl = decode_tile<MODE, BN>(p, t, tile_start, seg_off, nseg);
      const int acc = it % L::kAccBufs;
      const uint32_t aph = (uint32_t)(it / L::kAccBufs) & 1u;
      ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), aph, err, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint32_t t0 = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * 2 * BN);
      if (MODE == kGateUp) {
        const int ld = tl.shared ? p.Is : p.I;
        __nv_bfloat16 *out = tl.shared ? p.out_s : p.out;
        const int i = tl.rb * 128 + r;
        for (int c = 0; c < tl.N; c += 16) {
          float g[16], u[16];
          tmem_ld16(t0 + (uint32_t)c, g);
          tmem_ld16(t0 + (uint32_t)(BN + c), u);
          tmem_wait_ld();
          if (i < ld) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c + j < tl.ntok)
                out[(size_t)(tl.row0 + c + j) * ld + i] = __float2bfloat16_rn(silu_mul(g[j], u[j]));
          }
        }
      } else {
        __nv_bfloat16 *out = tl.shared ? p.out_s : p.out;
        const int ha = tl.rb * 256 + r, hb = ha + 128;
        for (int c = 0; c < tl.N; c += 16) {
          float va[16], vb[16];
          tmem_ld16(t0 + (uint32_t)c, va);
          tmem_ld16(t0 + (uint32_t)(BN + c), vb);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c + j < tl.ntok) {
              __nv_bfloat16 *row = out + (size_t)(tl.row0 + c + j) * p.H;
              if (ha < p.H) row[ha] = __float2bfloat16_rn(va[j]);
              if (hb < p.H) row[hb] = __float2bfloat16_rn(vb[j]);
            }
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
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
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
