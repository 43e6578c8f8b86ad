// Steps a5-a8: the grouped expert FFN -- gate/up GEMM through the route index,
// SiLU(gate) * up, down GEMM -- over uneven expert segments plus the shared
// expert as one more segment, in one persistent kernel on the 5th-generation
// tensor cores.
//
// "Hy3 Preview inference optimisation case", section 3 (FusedMoE): the gate-up
// GEMM reads the original input through the route index (no explicit gather
// copy); the down GEMM writes compactly per expert.  HunyuanImage 3.0 post:
// SwiGLU experts down(SiLU(gate(x)) * up(x)), stacked expert weights, the
// shared MLP applied to every token.
//
// Tiles.  Weight rows are the M = 128 operand of every MMA and the tokens of
// one expert chunk are the N operand (N = tokens rounded up to 16, at most
// BN <= 256).  A tile is 256 weight rows x N tokens: two MMAs per K step share
// one token tile and accumulate into two TMEM accumulators,
//   gate/up tile: D0 = gate rows i0..i0+127, D1 = up rows i0..i0+127, so gate
//                 row i and up row i land in the same TMEM lane and one thread
//                 forms SiLU(gate) * up -> bf16 activation A_act[p][i];
//   down tile:    D0 = w_down rows h0..h0+127, D1 = rows h0+128..h0+255 ->
//                 y[p][h].
// Sharing the token tile between 256 weight rows halves the token re-reads.
//
// Operand loads per 64-wide K step: the two 128-row weight boxes by TMA
// (128-byte swizzle); the token rows of a gate/up tile through the route index
// (token = perm[p] / k) by cp.async from 128 producer threads straight from
// `hidden`, written in the same swizzled layout (TMA's 4-row gather tops out
// far below the rate these tiles need); the activation rows of a down tile,
// which are contiguous, by at most four TMA boxes.
//
// Scheduling.  The tile list is every gate/up tile (per segment: 128-row
// blocks of I x token chunks, chunks innermost so they reuse the block's
// weights in L2) followed by every down tile.  CTAs (one per SM) claim tiles
// in that order from an atomic counter, so a down tile is claimed only after
// every gate/up tile has been claimed by a running CTA: its wait for the
// gate/up tiles of its segment (a per-segment completion count, bounded) can
// always be satisfied, whatever the residency of other CTAs.  Gate/up tiles
// never wait.  The last CTA to leave zeroes the counters for the next call.
//
// Pipelines.  Weights stream from HBM and need the longer lead; token rows
// come from L2.  So the two operands have rings of their own: kW weight slots
// (both 128-row boxes of one 64-wide K step, 32 KB) and kT token slots (N rows
// of one K step), each with full/empty barriers; the MMA of K step q takes
// weight slot q % kW and token slot q % kT.  Narrow tiles (decode) get six
// weight slots -- as many weight bytes in flight per SM as HBM needs -- 240-
// token tiles four, 256-token tiles three (fewer than three token slots
// starve the MMA).
//
// Warp roles: 0 (one thread) claims tiles and issues the weight TMA loads; 1-4
// load token rows (cp.async) or activation rows (TMA, one thread) and wait for
// a down tile's gate/up tiles; 5 issues the MMAs (one thread) and owns TMEM;
// 6-21 drain the accumulators, four warps per TMEM lane quarter taking its
// 16-column groups in turn (the epilogue of a wide tile is not overlapped with
// MMAs, so the more warps drain it the sooner TMEM is free: sixteen warps beat
// eight by 2-3 % on the wide tiles).  For BN <= 128 two TMEM accumulator pairs overlap one
// tile's epilogue with the next tile's MMAs (BN = 256 fills TMEM with one pair).
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"
#include "silu.cuh"

namespace moe {

namespace {

constexpr int kABytes = 2 * 128 * 128;  // weights of one K step: two 128-row x 64-bf16 boxes
constexpr int kMaxSeg = 258;            // E <= 256 routed + 1 shared (+1 sentinel)
constexpr int kWWarp = 0;               // tile claims + weight loads (lane 0)
constexpr int kTokWarp0 = 1;            // warps 1-4: token / activation loads
constexpr int kTokThreads = 128;
constexpr int kMmaWarp = 5;
constexpr int kEpiWarp0 = 6;            // warps 6.. : the epilogue
constexpr int kEpiWarps = 16;
constexpr int kGemmThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kWideEpiCols = 16;        // epilogue column group of tiles of 64 tokens or more
constexpr int kRing = 4;                // claimed tile ids in flight
// FP8 weights: TMA brings the E4M3 codes of a K step (two 128-row x 64-code
// boxes, 16 KB) into a ring of their own; eight converter warps (taking the
// place of eight epilogue warps) write them as bf16 into the weight slots
constexpr int kQBytes = 2 * 128 * 64;
constexpr int kCvtWarps = 8;
constexpr unsigned long long kDrainNs = 20000000ull;

// Ring depths: weight slots of 32 KB and token slots of BN x 128 bytes; with
// FP8 weights, code slots of 16 KB (the bytes in flight from HBM) and three
// bf16 weight slots between the converters and the MMAs.
template <int BN, bool Q8>
struct Rings {
  static constexpr int kW = Q8 ? 3 : BN >= 256 ? 3 : BN >= 240 ? 4 : BN >= 128 ? 5 : 6;
  static constexpr int kQ = Q8 ? (BN >= 128 ? 4 : 6) : 0;
  static constexpr int kT = BN >= 64 ? 3 : 4;
};

template <int BN, bool Q8>
struct Layout {
  static constexpr int kW = Rings<BN, Q8>::kW;
  static constexpr int kQ = Rings<BN, Q8>::kQ;
  static constexpr int kT = Rings<BN, Q8>::kT;
  static constexpr int kEpiW = Q8 ? kEpiWarps - kCvtWarps : kEpiWarps;  // epilogue warps
  static constexpr int kTokBytes = BN * 128;
  static constexpr int kQOff = kW * kABytes;
  static constexpr int kTOff = kQOff + kQ * kQBytes;
  // wide tiles stage each epilogue warp's 32-row x 16-token block in shared
  // memory and store whole 16-byte pieces of token rows (1 KB per warp)
  static constexpr bool kStageEpi = BN >= 256;
  static constexpr int kEpiOff = kTOff + kT * kTokBytes;
  static constexpr int kBarOff = kEpiOff + (kStageEpi ? kEpiW * kWideEpiCols * 64 : 0);  // tokens x 32 rows each
  // wfull, wempty per weight slot; tfull, tempty per token slot; acc full[2],
  // acc empty[2]; drain; id_full[kRing], id_empty[kRing]; qfull, qempty per code slot
  static constexpr int kNumBars = 2 * kW + 2 * kT + 5 + 2 * kRing + 2 * kQ;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;     // tmem slot, abort flag, ring of tile ids
  static constexpr int kStart1Off = kMiscOff + 64;
  static constexpr int kStart2Off = kStart1Off + 4 * kMaxSeg;
  static constexpr int kOffOff = kStart2Off + 4 * kMaxSeg;
  static constexpr int kBytes = kOffOff + 4 * kMaxSeg;
  static constexpr size_t kSmem = 1024 + kBytes;
  // accumulator pairs of 2 x BN columns: two while they fit in 512 columns, else one
  static constexpr int kAccBufs = 4 * BN <= 512 ? 2 : 1;
  static constexpr uint32_t kTmemUsed = kAccBufs * 2 * BN;
  // TMEM is allocated in powers of two columns
  static constexpr uint32_t kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128
                                        : kTmemUsed <= 256 ? 256 : 512;
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kTmemUsed <= 512, "TMEM budget");
  static_assert(kW <= 16 && kT <= 16 && kQ <= 16, "issue masks");
  static_assert(!Q8 || BN <= 128, "FP8 weights run the narrow tiles");
};

struct Tile {
  int phase;  // 0 gate/up, 1 down
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
__device__ __forceinline__ int seg_nrb(const GemmParams &p, int phase, bool shared) {
  if (phase == 0) return ((shared ? p.Is : p.I) + 127) >> 7;
  return (p.H + 255) >> 8;
}

__device__ __forceinline__ int seg_count(const GemmParams &p, const int *seg_off, int s) {
  return s == p.E ? p.T : seg_off[s + 1] - seg_off[s];
}

template <int BN>
__device__ __forceinline__ Tile decode_tile(const GemmParams &p, int t, const int *start1, const int *start2,
                                            const int *seg_off, int nseg) {
  Tile tl;
  tl.phase = t < start1[nseg] ? 0 : 1;
  const int *ts = tl.phase == 0 ? start1 : start2;
  const int u = tl.phase == 0 ? t : t - start1[nseg];
  int lo = 0, hi = nseg;  // ts[nseg] = total of the phase > u
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ts[mid] <= u) lo = mid;
    else hi = mid;
  }
  tl.seg = lo;
  tl.shared = (lo == p.E) ? 1 : 0;
  const int cnt = seg_count(p, seg_off, lo);
  const int nch = chunk_count<BN>(cnt);
  const int local = u - ts[lo];
  tl.rb = local / nch;
  const int ch = local - tl.rb * nch;
  const int base = chunk_base<BN>(cnt);
  const int pin = ch * base;
  tl.ntok = min(base, cnt - pin);
  tl.row0 = (tl.shared ? 0 : seg_off[lo]) + pin;
  tl.N = (tl.ntok + 15) & ~15;
  tl.nk = tl.phase == 0 ? (p.H >> 6) : ((tl.shared ? p.Is : p.I) >> 6);
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

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Eight E4M3 codes (two little-endian words, first code in the low byte) to the
// eight bf16 values they encode, exactly (every E4M3 value is a bf16 value; the
// row scale is applied to the fp32 accumulators in the epilogue instead).
__device__ __forceinline__ uint4 e4m3x8_to_bf16(uint32_t w0, uint32_t w1) {
  const uint32_t pr[4] = {w0 & 0xFFFFu, w0 >> 16, w1 & 0xFFFFu, w1 >> 16};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)pr[j], __NV_E4M3);
    const float2 f = __half22float2(__half2(hr));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    o[j] = *reinterpret_cast<const uint32_t *>(&b);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

template <int BN, bool Q8>
__global__ void __launch_bounds__(kGemmThreads, 1) expert_ffn_kernel(const __grid_constant__ GemmParams p) {
  using L = Layout<BN, Q8>;
  constexpr int KW = L::kW, KT = L::kT, KQ = L::kQ, EW = L::kEpiW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = (uint64_t *)(smem + L::kBarOff);
  uint32_t *tmem_slot = (uint32_t *)(smem + L::kMiscOff);
  volatile int *abort_flag = (volatile int *)(smem + L::kMiscOff + 4);
  volatile int *ring = (volatile int *)(smem + L::kMiscOff + 16);  // kRing claimed tile ids
  int *start1 = (int *)(smem + L::kStart1Off);
  int *start2 = (int *)(smem + L::kStart2Off);
  int *seg_off = (int *)(smem + L::kOffOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto wfull_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto wempty_bar = [&](int s) { return smem_u32(&bars[KW + s]); };
  auto tfull_bar = [&](int s) { return smem_u32(&bars[2 * KW + s]); };
  auto tempty_bar = [&](int s) { return smem_u32(&bars[2 * KW + KT + s]); };
  auto afull_bar = [&](int a) { return smem_u32(&bars[2 * KW + 2 * KT + a]); };
  auto aempty_bar = [&](int a) { return smem_u32(&bars[2 * KW + 2 * KT + 2 + a]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * KW + 2 * KT + 4]);
  auto id_full = [&](int r) { return smem_u32(&bars[2 * KW + 2 * KT + 5 + r]); };
  auto id_empty = [&](int r) { return smem_u32(&bars[2 * KW + 2 * KT + 5 + kRing + r]); };
  auto qfull_bar = [&](int s) { return smem_u32(&bars[2 * KW + 2 * KT + 5 + 2 * kRing + s]); };
  auto qempty_bar = [&](int s) { return smem_u32(&bars[2 * KW + 2 * KT + 5 + 2 * kRing + KQ + s]); };
  auto q_smem = [&](int s) { return smem_u32(smem + L::kQOff + s * kQBytes); };
  auto w_smem = [&](int s) { return smem_u32(smem + s * kABytes); };
  auto t_smem = [&](int s) { return smem_u32(smem + L::kTOff + s * L::kTokBytes); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < KW; ++s) {
      mbar_init(wfull_bar(s), Q8 ? kCvtWarps : 1);  // the weight loader's expect_tx arrival, or the converters
      mbar_init(wempty_bar(s), 1);                  // MMA commit
    }
    for (int s = 0; s < KQ; ++s) {
      mbar_init(qfull_bar(s), 1);           // the loader's expect_tx arrival
      mbar_init(qempty_bar(s), kCvtWarps);  // converters done reading
    }
    for (int s = 0; s < KT; ++s) {
      mbar_init(tfull_bar(s), kTokThreads);  // one arrival per loader thread (cp.async, or the TMA expect_tx)
      mbar_init(tempty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(afull_bar(a), 1);
      mbar_init(aempty_bar(a), EW);
    }
    mbar_init(drain_bar, 1);
    for (int r = 0; r < kRing; ++r) {
      mbar_init(id_full(r), 1);
      mbar_init(id_empty(r), 1 + 4 + EW + (Q8 ? kCvtWarps : 0));  // MMA, token loaders, epilogue, converters
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWWarp && lane == 0) {  // only the maps of the phases this launch runs are filled in
    if (p.phases & 1) {
      tma_prefetch_desc(&p.map_wg);
      tma_prefetch_desc(&p.map_wu);
    }
    if (p.phases & 2) tma_prefetch_desc(&p.map_wd);
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

  // ---------------- tile lists of both phases from the expert offsets (one warp)
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
#pragma unroll
    for (int ph = 0; ph < 2; ++ph) {
      int *ts = ph == 0 ? start1 : start2;
      const bool on = good && (p.phases >> ph) & 1;
      int local = 0;
      for (int s = s0; s < min(nseg, s0 + per); ++s)
        local += on ? chunk_count<BN>(seg_count(p, seg_off, s)) * seg_nrb(p, ph, s == p.E) : 0;
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      int run = incl - local;
      for (int s = s0; s < min(nseg, s0 + per); ++s) {
        ts[s] = run;
        run += on ? chunk_count<BN>(seg_count(p, seg_off, s)) * seg_nrb(p, ph, s == p.E) : 0;
      }
      if (lane == 31) ts[nseg] = incl;
    }
  }
  __syncthreads();
  const int total = start1[nseg] + start2[nseg];
  unsigned *err = p.err;
  unsigned *claim = p.sync + kSyncClaim;
  unsigned *done1 = p.sync + kSyncDone;  // gate/up tiles finished, per segment
  bool ok = true;

  if (warp == kWWarp) {
    // ================= tile claims and weight loads (one thread); FP8 weights
    // go to the code slots, bf16 weights straight to the weight slots
    if (lane == 0) {
      constexpr int NS = Q8 ? KQ : KW;
      const uint64_t pol_w = policy_evict_first();
      int ws = 0;
      uint32_t wph = 0;
      uint32_t issued = 0, issued_par = 0;  // per weight slot: a load issued, and its phase parity
      for (int i = 0; ok; ++i) {
        const int r = i % kRing;
        ok = mbar_wait(id_empty(r), ((uint32_t)(i / kRing) & 1u) ^ 1u, err, abort_flag);
        if (!ok) break;
        const int t0 = (int)atomicAdd(claim, 1u);
        const int t = t0 < total ? t0 : -1;
        ring[r] = t;
        mbar_arrive(id_full(r));
        if (t < 0) break;
        const Tile tl = decode_tile<BN>(p, t, start1, start2, seg_off, nseg);
        const int i0 = tl.rb * (tl.phase == 0 ? 128 : 256);
        for (int kb = 0; kb < tl.nk; ++kb) {
          const uint32_t fb = Q8 ? qfull_bar(ws) : wfull_bar(ws);
          ok = mbar_wait(Q8 ? qempty_bar(ws) : wempty_bar(ws), wph ^ 1u, err, abort_flag);
          if (!ok) break;
          const int k0 = kb * 64;
          mbar_arrive_expect_tx(fb, (uint32_t)(Q8 ? kQBytes : kABytes));
          issued |= 1u << ws;
          issued_par = (issued_par & ~(1u << ws)) | (wph << ws);
          const uint32_t a0 = Q8 ? q_smem(ws) : w_smem(ws), a1 = a0 + (Q8 ? kQBytes / 2 : kABytes / 2);
          if (tl.phase == 0) {
            if (tl.shared) {
              tma_load_2d_hint(a0, &p.map_sg, fb, k0, i0, pol_w);
              tma_load_2d_hint(a1, &p.map_su, fb, k0, i0, pol_w);
            } else {
              tma_load_3d_hint(a0, &p.map_wg, fb, k0, i0, tl.seg, pol_w);
              tma_load_3d_hint(a1, &p.map_wu, fb, k0, i0, tl.seg, pol_w);
            }
          } else {
            if (tl.shared) {
              tma_load_2d_hint(a0, &p.map_sd, fb, k0, i0, pol_w);
              tma_load_2d_hint(a1, &p.map_sd, fb, k0, i0 + 128, pol_w);
            } else {
              tma_load_3d_hint(a0, &p.map_wd, fb, k0, i0, tl.seg, pol_w);
              tma_load_3d_hint(a1, &p.map_wd, fb, k0, i0 + 128, tl.seg, pol_w);
            }
          }
          if (++ws == NS) {
            ws = 0;
            wph ^= 1u;
          }
        }
      }
      if (!ok)
        for (int s = 0; s < NS; ++s)
          if ((issued >> s) & 1u) mbar_wait_drain(Q8 ? qfull_bar(s) : wfull_bar(s), (issued_par >> s) & 1u);
    }
  } else if (warp < kTokWarp0 + 4) {
    // ================= token rows (gate/up) or activation rows (down)
    const int tid = threadIdx.x - 32 * kTokWarp0;  // 0..127
    const int c8 = tid & 7, rbase = tid >> 3;
    int ts = 0;
    uint32_t tph = 0;
    uint32_t issued = 0, issued_par = 0;  // per token slot: an activation TMA issued (thread 0)
    for (int i = 0; ok; ++i) {
      const int r = i % kRing;
      ok = __all_sync(0xffffffffu, mbar_wait(id_full(r), (uint32_t)(i / kRing) & 1u, err, abort_flag));
      if (!ok) break;
      const int t = ring[r];
      __syncwarp();
      if (lane == 0) mbar_arrive(id_empty(r));
      if (t < 0) break;
      const Tile tl = decode_tile<BN>(p, t, start1, start2, seg_off, nseg);

      // ---- a down tile needs every gate/up tile of its segment
      if (tl.phase == 1 && (p.phases & 1) && tid == 0) {
        const unsigned need = (unsigned)(chunk_count<BN>(seg_count(p, seg_off, tl.seg)) * seg_nrb(p, 0, tl.shared));
        if (ld_acquire_gpu(done1 + tl.seg) < need) {
          const unsigned long long t0 = globaltimer();
          while (ld_acquire_gpu(done1 + tl.seg) < need) {
            if (*abort_flag || globaltimer() - t0 > kWaitLimitNs) {
              if (!*abort_flag && err != nullptr) atomicOr(err, MOE_DEVERR_TIMEOUT);
              *abort_flag = 1;
              break;
            }
            __nanosleep(64);
          }
        }
        fence_proxy_async_global();  // the activations were written by other CTAs' generic stores
      }

      // ---- token rows of this thread for a gate/up tile: rows rbase + 16 j
      const __nv_bfloat16 *src[BN / 16];
      if (tl.phase == 0) {
        bool bad = false;
#pragma unroll
        for (int j = 0; j < BN / 16; ++j) {
          const int row = rbase + 16 * j;
          const int rr = row < tl.ntok ? row : 0;
          int tok = 0;
          if (row < tl.N) {
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
      for (int kb = 0; kb < tl.nk; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(tempty_bar(ts), tph ^ 1u, err, abort_flag));
        if (!ok || *abort_flag) {
          ok = false;
          break;
        }
        const int k0 = kb * 64;
        const uint32_t bs = t_smem(ts);
        if (tl.phase == 0) {
#pragma unroll
          for (int j = 0; j < BN / 16; ++j) {
            const int row = rbase + 16 * j;
            if (row < tl.N) cp_async_16(bs + row * 128 + ((c8 ^ (row & 7)) << 4), src[j] + k0);
          }
          cp_async_arrive_noinc(tfull_bar(ts));
        } else if (tid == 0) {
          // activation rows row0 .. row0 + N (contiguous, N a multiple of 16 and
          // <= 256): boxes of 128 rows while they fit, then one each of 64/32/16
          mbar_arrive_expect_tx(tfull_bar(ts), (uint32_t)(tl.N * 128));
          issued |= 1u << ts;
          issued_par = (issued_par & ~(1u << ts)) | (tph << ts);
          const CUtensorMap *mb = tl.shared ? p.map_acts : p.map_act;
          int off = 0;
          while (tl.N - off >= 128) {
            tma_load_2d(bs + (uint32_t)off * 128, &mb[3], tfull_bar(ts), k0, tl.row0 + off);
            off += 128;
          }
#pragma unroll
          for (int bi = 2; bi >= 0; --bi) {
            const int h = 16 << bi;
            if (tl.N - off >= h) {
              tma_load_2d(bs + (uint32_t)off * 128, &mb[bi], tfull_bar(ts), k0, tl.row0 + off);
              off += h;
            }
          }
        } else {
          mbar_arrive(tfull_bar(ts));
        }
        if (++ts == KT) {
          ts = 0;
          tph ^= 1u;
        }
      }
    }
    if (!ok) {
      cp_async_wait_all();
      if (tid == 0)
        for (int s = 0; s < KT; ++s)
          if ((issued >> s) & 1u) mbar_wait_drain(tfull_bar(s), (issued_par >> s) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // ================= MMA issuer
    if (lane == 0) {
      int ws = 0, ts = 0;
      uint32_t wph = 0, tph = 0;
      bool any = false;
      for (int i = 0; ok; ++i) {
        const int r = i % kRing;
        ok = mbar_wait(id_full(r), (uint32_t)(i / kRing) & 1u, err, abort_flag);
        if (!ok) break;
        const int t = ring[r];
        mbar_arrive(id_empty(r));
        if (t < 0) break;
        const Tile tl = decode_tile<BN>(p, t, start1, start2, seg_off, nseg);
        const int acc = i % L::kAccBufs;
        const uint32_t aph = (uint32_t)(i / L::kAccBufs) & 1u;
        ok = mbar_wait(aempty_bar(acc), aph ^ 1u, err, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)(acc * 2 * BN);
        const uint32_t d1 = d0 + (uint32_t)BN;
        const uint32_t idesc = idesc_bf16(128, tl.N);
        for (int kb = 0; kb < tl.nk; ++kb) {
          ok = mbar_wait(wfull_bar(ws), wph, err, abort_flag) && mbar_wait(tfull_bar(ts), tph, err, abort_flag);
          if (!ok) break;
          if (tl.phase == 0) fence_proxy_async_smem();  // token rows were written by cp.async
          tc_fence_after();
          const uint64_t a0 = sdesc_sw128(w_smem(ws));
          const uint64_t a1 = sdesc_sw128(w_smem(ws) + 16384);
          const uint64_t bd = sdesc_sw128(t_smem(ts));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            umma_bf16(d0, a0 + 2 * kk, bd + 2 * kk, idesc, accum);
            umma_bf16(d1, a1 + 2 * kk, bd + 2 * kk, idesc, accum);
          }
          any = true;
          umma_commit(wempty_bar(ws));
          umma_commit(tempty_bar(ts));
          if (++ws == KW) {
            ws = 0;
            wph ^= 1u;
          }
          if (++ts == KT) {
            ts = 0;
            tph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(afull_bar(acc));
      }
      if (!ok && any) {
        umma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0);
      }
    }
  } else if (warp < kEpiWarp0 + EW) {
    // ================= epilogue (warps 6..21 -> TMEM lane quarters 2,3,0,1, four times;
    // with FP8 weights warps 6..13, twice)
    const int q = warp & 3;
    // column groups of kEpiCols (16: one TMEM wait per 16 columns);
    // the warps of a lane quarter take its groups in turn
    constexpr int kEpiCols = BN >= 64 ? kWideEpiCols : 16;
    constexpr int kEpiStep = kEpiCols * (EW / 4);  // the lane quarter's warps take groups in turn
    const int c_first = kEpiCols * ((warp - kEpiWarp0) >> 2);
    __nv_bfloat16 *stage = reinterpret_cast<__nv_bfloat16 *>(smem + L::kEpiOff + (warp - kEpiWarp0) * kEpiCols * 64);
    const int r = 32 * q + lane;  // weight row within the 128-row half
    for (int i = 0; ok; ++i) {
      const int rs = i % kRing;
      ok = __all_sync(0xffffffffu, mbar_wait(id_full(rs), (uint32_t)(i / kRing) & 1u, err, abort_flag));
      if (!ok) break;
      const int t = ring[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(id_empty(rs));
      if (t < 0) break;
      const Tile tl = decode_tile<BN>(p, t, start1, start2, seg_off, nseg);
      const int acc = i % L::kAccBufs;
      const uint32_t aph = (uint32_t)(i / L::kAccBufs) & 1u;
      ok = __all_sync(0xffffffffu, mbar_wait(afull_bar(acc), aph, err, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint32_t t0 = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * 2 * BN);
      // FP8 weights: the accumulators hold sum(value(code) * x); this lane's
      // row scales turn them into the products with the weights
      float s0 = 1.0f, s1 = 1.0f;
      if constexpr (Q8) {
        if (tl.phase == 0) {
          const int ii = tl.rb * 128 + r;
          if (ii < (tl.shared ? p.Is : p.I)) {
            s0 = __ldg((tl.shared ? p.sc_sg : p.sc_g + (size_t)tl.seg * p.I) + ii);
            s1 = __ldg((tl.shared ? p.sc_su : p.sc_u + (size_t)tl.seg * p.I) + ii);
          }
        } else {
          const int ha = tl.rb * 256 + r, hb = ha + 128;
          const float *sp = tl.shared ? p.sc_sd : p.sc_d + (size_t)tl.seg * p.H;
          if (ha < p.H) s0 = __ldg(sp + ha);
          if (hb < p.H) s1 = __ldg(sp + hb);
        }
      }
      if constexpr (L::kStageEpi) {
        // lane j of the warp owns weight row first + j; a group of ncol tokens is
        // written to the staging block as [token][32 rows] bf16, then each lane
        // stores 16 bytes (8 rows of one token): 4 lanes per token row piece.
        // y goes out with the streaming (evict-first) hint: it is read only by
        // the combine after this kernel, while the activations are re-read
        // here by the down tiles and should stay in L2.
        auto flush = [&](__nv_bfloat16 *rows, size_t ld, int first, int limit, int c, int ncol, bool stream) {
          __syncwarp();
          for (int pass = 0; pass < ncol / 8; ++pass) {
            const int jj = pass * 8 + (lane >> 2), qq = lane & 3;
            const uint4 v = *reinterpret_cast<const uint4 *>(stage + jj * 32 + qq * 8);
            if (c + jj < tl.ntok && first + qq * 8 < limit) {
              uint4 *dst = reinterpret_cast<uint4 *>(rows + (size_t)(c + jj) * ld + first + qq * 8);
              if (stream) __stcs(dst, v);
              else *dst = v;
            }
          }
          __syncwarp();
        };
        if (tl.phase == 0) {
          const int ld = tl.shared ? p.Is : p.I;
          __nv_bfloat16 *rows = (tl.shared ? p.act_s : p.act) + (size_t)tl.row0 * ld;
          const int first = tl.rb * 128 + 32 * q;
          for (int c = c_first; c < tl.N; c += kEpiStep) {
            float g[32], u[32];
            const int ncol = min(kEpiCols, tl.N - c);
            if (ncol == 32) {
              tmem_ld32(t0 + (uint32_t)c, g);
              tmem_ld32(t0 + (uint32_t)(BN + c), u);
            } else {
              tmem_ld16_lo(t0 + (uint32_t)c, g);
              tmem_ld16_lo(t0 + (uint32_t)(BN + c), u);
            }
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < ncol) stage[j * 32 + lane] = __float2bfloat16_rn(silu_mul(g[j], u[j]));
            flush(rows, (size_t)ld, first, ld, c, ncol, false);
          }
        } else {
          __nv_bfloat16 *rows = (tl.shared ? p.y_s : p.y) + (size_t)tl.row0 * p.H;
          const int first = tl.rb * 256 + 32 * q;
          for (int c = c_first; c < tl.N; c += kEpiStep) {
            float va[32], vb[32];
            const int ncol = min(kEpiCols, tl.N - c);
            if (ncol == 32) {
              tmem_ld32(t0 + (uint32_t)c, va);
              tmem_ld32(t0 + (uint32_t)(BN + c), vb);
            } else {
              tmem_ld16_lo(t0 + (uint32_t)c, va);
              tmem_ld16_lo(t0 + (uint32_t)(BN + c), vb);
            }
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < ncol) stage[j * 32 + lane] = __float2bfloat16_rn(va[j]);
            flush(rows, (size_t)p.H, first, p.H, c, ncol, true);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < ncol) stage[j * 32 + lane] = __float2bfloat16_rn(vb[j]);
            flush(rows, (size_t)p.H, first + 128, p.H, c, ncol, true);
          }
        }
      } else if (tl.phase == 0) {
        const int ld = tl.shared ? p.Is : p.I;
        __nv_bfloat16 *out = tl.shared ? p.act_s : p.act;
        const int ii = tl.rb * 128 + r;
        for (int c = c_first; c < tl.N; c += kEpiStep) {
          if (kEpiCols == 32 && c + 32 <= tl.N) {
            float g[32], u[32];
            tmem_ld32(t0 + (uint32_t)c, g);
            tmem_ld32(t0 + (uint32_t)(BN + c), u);
            tmem_wait_ld();
            if (ii < ld) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (c + j < tl.ntok)
                  out[(size_t)(tl.row0 + c + j) * ld + ii] =
                      __float2bfloat16_rn(Q8 ? silu_mul(g[j] * s0, u[j] * s1) : silu_mul(g[j], u[j]));
            }
          } else {
            for (int c16 = c; c16 < min(c + kEpiCols, tl.N); c16 += 16) {
              float g[16], u[16];
              tmem_ld16(t0 + (uint32_t)c16, g);
              tmem_ld16(t0 + (uint32_t)(BN + c16), u);
              tmem_wait_ld();
              if (ii < ld) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (c16 + j < tl.ntok)
                    out[(size_t)(tl.row0 + c16 + j) * ld + ii] =
                        __float2bfloat16_rn(Q8 ? silu_mul(g[j] * s0, u[j] * s1) : silu_mul(g[j], u[j]));
              }
            }
          }
        }
      } else {
        __nv_bfloat16 *out = tl.shared ? p.y_s : p.y;
        const int ha = tl.rb * 256 + r, hb = ha + 128;
        for (int c = c_first; c < tl.N; c += kEpiStep) {
          if (kEpiCols == 32 && c + 32 <= tl.N) {
            float va[32], vb[32];
            tmem_ld32(t0 + (uint32_t)c, va);
            tmem_ld32(t0 + (uint32_t)(BN + c), vb);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (c + j < tl.ntok) {
                __nv_bfloat16 *row = out + (size_t)(tl.row0 + c + j) * p.H;
                if (ha < p.H) __stcs(row + ha, __float2bfloat16_rn(Q8 ? va[j] * s0 : va[j]));
                if (hb < p.H) __stcs(row + hb, __float2bfloat16_rn(Q8 ? vb[j] * s1 : vb[j]));
              }
            }
          } else {
            for (int c16 = c; c16 < min(c + kEpiCols, tl.N); c16 += 16) {
              float va[16], vb[16];
              tmem_ld16(t0 + (uint32_t)c16, va);
              tmem_ld16(t0 + (uint32_t)(BN + c16), vb);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                if (c16 + j < tl.ntok) {
                  __nv_bfloat16 *row = out + (size_t)(tl.row0 + c16 + j) * p.H;
                  if (ha < p.H) __stcs(row + ha, __float2bfloat16_rn(Q8 ? va[j] * s0 : va[j]));
                  if (hb < p.H) __stcs(row + hb, __float2bfloat16_rn(Q8 ? vb[j] * s1 : vb[j]));
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty_bar(acc));
      if (tl.phase == 0 && (p.phases & 2)) {
        // publish: this gate/up tile's activations are written (release to the down tiles)
        __threadfence();
        named_bar_sync(2, 32 * EW);
        if (warp == kEpiWarp0 && lane == 0) atomicAdd(done1 + tl.seg, 1u);
      }
    }
  } else if constexpr (Q8) {
    // ================= FP8 weights (warps 14..21): codes -> bf16 weight slots
    // (the values of the codes; the epilogue applies each row's scale).
    // Converter warp cw takes rows 32 (cw & 3) .. + 31 of box cw >> 2; per
    // pass, lane l converts 16 codes (chunk l & 3) of row 8 it + (l >> 2), so a
    // warp reads 512 contiguous bytes and writes whole 128-byte swizzled rows.
    const int cw = warp - (kEpiWarp0 + EW);
    const int box = cw >> 2, c = lane & 3;
    int ws = 0, qs = 0;
    uint32_t wph = 0, qph = 0;
    for (int i = 0; ok; ++i) {
      const int rs = i % kRing;
      ok = __all_sync(0xffffffffu, mbar_wait(id_full(rs), (uint32_t)(i / kRing) & 1u, err, abort_flag));
      if (!ok) break;
      const int t = ring[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(id_empty(rs));
      if (t < 0) break;
      const Tile tl = decode_tile<BN>(p, t, start1, start2, seg_off, nseg);
      for (int kb = 0; kb < tl.nk; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(qfull_bar(qs), qph, err, abort_flag) &&
                                         mbar_wait(wempty_bar(ws), wph ^ 1u, err, abort_flag));
        if (!ok) break;
        const uint8_t *src = smem + L::kQOff + qs * kQBytes + box * (kQBytes / 2);
        uint8_t *dst = smem + ws * kABytes + box * (kABytes / 2);
        uint4 v[4];  // every read first: the stores cannot then hold back the next loads
#pragma unroll
        for (int it = 0; it < 4; ++it)
          v[it] = *reinterpret_cast<const uint4 *>(src + (32 * (cw & 3) + 8 * it + (lane >> 2)) * 64 + c * 16);
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int rr = 32 * (cw & 3) + 8 * it + (lane >> 2);
          *reinterpret_cast<uint4 *>(dst + rr * 128 + (((2 * c) ^ (rr & 7)) << 4)) = e4m3x8_to_bf16(v[it].x, v[it].y);
          *reinterpret_cast<uint4 *>(dst + rr * 128 + (((2 * c + 1) ^ (rr & 7)) << 4)) =
              e4m3x8_to_bf16(v[it].z, v[it].w);
        }
        fence_proxy_async_smem();  // generic-proxy writes read by the tensor core
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(wfull_bar(ws));
          mbar_arrive(qempty_bar(qs));
        }
        if (++ws == KW) {
          ws = 0;
          wph ^= 1u;
        }
        if (++qs == KQ) {
          qs = 0;
          qph ^= 1u;
        }
      }
    }
  }

  __syncwarp();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  // the last CTA out zeroes the claim counter and the completion counts
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(p.sync + kSyncExit, 1u);
    if (prev == gridDim.x - 1) {
      volatile unsigned *s = p.sync;
      s[kSyncClaim] = 0;
      for (int i = 0; i < nseg; ++i) s[kSyncDone + i] = 0;
      __threadfence();
      s[kSyncExit] = 0;
    }
  }
}

// Widest tile for a batch.  Past 128 tokens: 256 when experts average more
// than 256 tokens (fewer chunks, so fewer passes over each expert's weights),
// else 240, whose smaller token slots leave room for a fourth weight slot --
// more weight bytes in flight for the many one-chunk experts.
int gemm_tile_n(int T, int top_k, int E) {
  if (T <= 16) return 16;
  if (T <= 32) return 32;
  if (T <= 64) return 64;
  if (T <= 128) return 128;
  return (long long)T * top_k > 256LL * E ? 256 : 240;
}

namespace {
template <int BN, bool Q8>
cudaError_t launch_one(const GemmParams &p, int num_ctas, cudaStream_t stream, bool pdl) {
  using L = Layout<BN, Q8>;
  static thread_local unsigned long long attr_ctx = 0;
  const cudaError_t e = set_smem_attr_once((const void *)expert_ffn_kernel<BN, Q8>, (int)L::kSmem, attr_ctx);
  if (e != cudaSuccess) return e;
  void *args[] = {(void *)&p};
  return launch_ex((const void *)expert_ffn_kernel<BN, Q8>, dim3(num_ctas), dim3(kGemmThreads), L::kSmem, stream, pdl, 1,
                   args);
}
}  // namespace

cudaError_t launch_expert_ffn(const GemmParams &p, int bn, int num_ctas, cudaStream_t stream, bool pdl) {
  if (p.q8) {  // FP8 weights: narrow tiles only (the code ring takes the shared memory of wide token slots)
    switch (bn < 128 ? bn : 128) {
      case 16: return launch_one<16, true>(p, num_ctas, stream, pdl);
      case 32: return launch_one<32, true>(p, num_ctas, stream, pdl);
      case 64: return launch_one<64, true>(p, num_ctas, stream, pdl);
      case 128: return launch_one<128, true>(p, num_ctas, stream, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 16: return launch_one<16, false>(p, num_ctas, stream, pdl);
    case 32: return launch_one<32, false>(p, num_ctas, stream, pdl);
    case 64: return launch_one<64, false>(p, num_ctas, stream, pdl);
    case 128: return launch_one<128, false>(p, num_ctas, stream, pdl);
    case 240: return launch_one<240, false>(p, num_ctas, stream, pdl);
    case 256: return launch_one<256, false>(p, num_ctas, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
