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
// Tiles.  Weight rows are the M operand of every MMA and the tokens of one
// expert chunk are the N operand (at most BN <= 256).  Two MMAs per K step
// share one token tile and accumulate into two TMEM accumulators:
//   gate/up tile: D0 = gate rows, D1 = the up rows of the same indices, so gate
//                 row i and up row i land in the same TMEM lane and one thread
//                 forms SiLU(gate) * up -> bf16 activation A_act[p][i];
//   down tile:    D0, D1 = two blocks of w_down rows -> y[p][h].
// Narrow tiles (BN <= 128, small batches) run one CTA per tile with M = 128:
// 128 gate + 128 up rows, or 256 down rows.  256-token tiles run on CTA pairs
// (clusters of two) with the 2-SM MMA, M = 256: the pair's tile is 256 gate +
// 256 up rows (512 down rows) x N tokens; each CTA holds its 128 rows of every
// weight block and half of the token rows, and the first CTA's MMAs read the
// other half from its partner's shared memory.  Per SM that is 48 KB of
// operands per K step instead of 64 KB for the same tensor work -- the bytes
// that enter each SM are what bound these tiles.
//
// Operand loads per 64-wide K step: the 128-row weight boxes by TMA (128-byte
// swizzle); the token rows of a gate/up tile through the route index (token =
// perm[p] / k) by cp.async from 128 threads straight from `hidden`, written in
// the same swizzled layout (TMA's 4-row gather tops out far below the rate
// these tiles need); the activation rows of a down tile, which are contiguous,
// by at most four TMA boxes.
//
// Scheduling.  The tile list is every gate/up tile (per segment: row blocks x
// token chunks, chunks innermost so they reuse the block's weights in L2)
// followed by every down tile.  CTAs (one per SM; pairs claim through their
// first CTA) claim tiles in that order from an atomic counter, so a down tile
// is claimed only after every gate/up tile has been claimed by a running CTA:
// its wait for the gate/up tiles of its segment (a per-segment completion
// count, bounded) can always be satisfied, whatever the residency of other
// CTAs.  Gate/up tiles never wait.  The last CTA to leave zeroes the counters.
//
// Pipelines.  The two operands have rings of their own: kW weight slots (both
// 128-row boxes of one K step, 32 KB) and kT token slots (the CTA's token rows
// of one K step), each with full/empty barriers; the MMA of K step q takes
// weight slot q % kW and token slot q % kT.  In a pair the first CTA's MMA
// thread also waits for the partner's slots: the partner's otherwise idle MMA
// thread relays their completion with an asynchronous 4-byte store into the
// first CTA that completes a transaction on a third ring of barriers (a plain
// remote arrive with cluster-scope release blocks the relaying thread for more
// than a K step of MMAs), and the MMA commits release the slots of both CTAs.
//
// Warp roles: 0 (one thread) claims tiles and issues the weight TMA loads; 1-4
// load token rows (cp.async) or activation rows (TMA, one thread) and wait for
// a down tile's gate/up tiles; 5 issues the MMAs (one thread; in a pair's
// second CTA it relays) and owns TMEM; 6-13 drain the accumulators, two warps
// per TMEM lane quarter on alternate column groups.  For BN <= 128 two TMEM
// accumulator pairs overlap one tile's epilogue with the next tile's MMAs.
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kABytes = 2 * 128 * 128;  // weights of one K step: two 128-row x 64-bf16 boxes
constexpr int kMaxSeg = 258;            // E <= 256 routed + 1 shared (+1 sentinel)
constexpr int kWWarp = 0;               // tile claims + weight loads (lane 0)
constexpr int kTokWarp0 = 1;            // warps 1-4: token / activation loads
constexpr int kTokThreads = 128;
constexpr int kMmaWarp = 5;
constexpr int kEpiWarp0 = 6;            // warps 6.. : the epilogue
constexpr int kEpiWarps = 8;
constexpr int kGemmThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kWideEpiCols = 32;        // epilogue column group of tiles of 64 tokens or more
constexpr int kRing = 4;                // claimed tile ids in flight
constexpr uint16_t kBoth = 3;           // cluster mask of a CTA pair
constexpr unsigned long long kDrainNs = 20000000ull;

// Ring depths: weight slots of 32 KB, token slots of the CTA's token rows.
template <int BN, bool PAIR>
struct Rings {
  static constexpr int kW = PAIR ? 4 : BN >= 256 ? 3 : BN >= 128 ? 5 : 6;
  static constexpr int kT = PAIR ? 4 : BN >= 256 ? 3 : BN >= 64 ? 3 : 4;
};

template <int BN, bool PAIR>
struct Layout {
  static constexpr int kW = Rings<BN, PAIR>::kW;
  static constexpr int kT = Rings<BN, PAIR>::kT;
  static constexpr int kTokRows = PAIR ? BN / 2 : BN;  // token rows a CTA holds per K step
  static constexpr int kTokBytes = kTokRows * 128;
  static constexpr int kTOff = kW * kABytes;
  // wide tiles stage each epilogue warp's 32-row x 32-token block in shared
  // memory and store whole 16-byte pieces of token rows (2 KB per warp)
  static constexpr bool kStageEpi = BN >= 256;
  static constexpr int kEpiOff = kTOff + kT * kTokBytes;
  static constexpr int kBarOff = kEpiOff + (kStageEpi ? kEpiWarps * kWideEpiCols * 64 : 0);
  // wfull, wempty per weight slot; tfull, tempty, pfull (partner ready) per
  // token slot; acc full[2], acc empty[2]; drain; id_full[kRing], id_empty[kRing]
  static constexpr int kNumBars = 2 * kW + 3 * kT + 5 + 2 * kRing;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;  // tmem slot, abort flag, ring of tile ids, relay words
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
  static_assert(kW <= 16 && kT <= 8, "issue masks, relay words");
  static_assert(!PAIR || BN == 256, "CTA pairs run the 256-token tiles");
};

struct Tile {
  int phase;  // 0 gate/up, 1 down
  int seg, rb, row0, ntok, N, nk, shared;
};

// Tokens per chunk for a segment of `cnt` tokens: the fewest chunks of at most
// BN tokens, made as even as possible and rounded up to 16 (32 for a pair,
// whose CTAs hold half each).
template <int BN, bool PAIR>
__device__ __forceinline__ int chunk_base(int cnt) {
  constexpr int q = PAIR ? 32 : 16;
  const int n0 = (cnt + BN - 1) / BN;
  const int per = (cnt + n0 - 1) / n0;
  return (per + q - 1) & ~(q - 1);
}
template <int BN, bool PAIR>
__device__ __forceinline__ int chunk_count(int cnt) {
  if (cnt <= 0) return 0;
  const int b = chunk_base<BN, PAIR>(cnt);
  return (cnt + b - 1) / b;
}

// Weight rows of a tile: gate/up 128 (pair: 256) gate/up row pairs; down 256
// (pair: 512) rows of w_down.
template <bool PAIR>
__device__ __forceinline__ int tile_rows(int phase) {
  return (phase == 0 ? 128 : 256) * (PAIR ? 2 : 1);
}
template <bool PAIR>
__device__ __forceinline__ int seg_nrb(const GemmParams &p, int phase, bool shared) {
  const int rows = phase == 0 ? (shared ? p.Is : p.I) : p.H;
  return (rows + tile_rows<PAIR>(phase) - 1) / tile_rows<PAIR>(phase);
}

__device__ __forceinline__ int seg_count(const GemmParams &p, const int *seg_off, int s) {
  return s == p.E ? p.T : seg_off[s + 1] - seg_off[s];
}

template <int BN, bool PAIR>
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
  const int nch = chunk_count<BN, PAIR>(cnt);
  const int local = u - ts[lo];
  tl.rb = local / nch;
  const int ch = local - tl.rb * nch;
  const int base = chunk_base<BN, PAIR>(cnt);
  const int pin = ch * base;
  tl.ntok = min(base, cnt - pin);
  tl.row0 = (tl.shared ? 0 : seg_off[lo]) + pin;
  tl.N = PAIR ? (tl.ntok + 31) & ~31 : (tl.ntok + 15) & ~15;
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

// SiLU(g) * u with the fast reciprocal-based division: the result is rounded
// to bf16, far coarser than the division's few-ulp error, and for g < -87 the
// denominator overflows and the quotient goes to zero, which is SiLU's limit.
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

}  // namespace

template <int BN, bool PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1) expert_ffn_kernel(const __grid_constant__ GemmParams p) {
  using L = Layout<BN, PAIR>;
  constexpr int KW = L::kW, KT = L::kT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = (uint64_t *)(smem + L::kBarOff);
  uint32_t *tmem_slot = (uint32_t *)(smem + L::kMiscOff);
  volatile int *abort_flag = (volatile int *)(smem + L::kMiscOff + 4);
  volatile int *ring = (volatile int *)(smem + L::kMiscOff + 16);  // kRing claimed tile ids
  uint32_t *relay_word = (uint32_t *)(smem + L::kMiscOff + 32);    // pair: one per token slot (<= 8)
  int *start1 = (int *)(smem + L::kStart1Off);
  int *start2 = (int *)(smem + L::kStart2Off);
  int *seg_off = (int *)(smem + L::kOffOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = PAIR ? (int)cluster_ctarank() : 0;  // 0: the pair's MMA-issuing CTA
  auto wfull_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto wempty_bar = [&](int s) { return smem_u32(&bars[KW + s]); };
  auto tfull_bar = [&](int s) { return smem_u32(&bars[2 * KW + s]); };
  auto tempty_bar = [&](int s) { return smem_u32(&bars[2 * KW + KT + s]); };
  auto pfull_bar = [&](int s) { return smem_u32(&bars[2 * KW + 2 * KT + s]); };
  auto afull_bar = [&](int a) { return smem_u32(&bars[2 * KW + 3 * KT + a]); };
  auto aempty_bar = [&](int a) { return smem_u32(&bars[2 * KW + 3 * KT + 2 + a]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * KW + 3 * KT + 4]);
  auto id_full = [&](int r) { return smem_u32(&bars[2 * KW + 3 * KT + 5 + r]); };
  auto id_empty = [&](int r) { return smem_u32(&bars[2 * KW + 3 * KT + 5 + kRing + r]); };
  auto w_smem = [&](int s) { return smem_u32(smem + s * kABytes); };
  auto t_smem = [&](int s) { return smem_u32(smem + L::kTOff + s * L::kTokBytes); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < KW; ++s) {
      mbar_init(wfull_bar(s), 1);   // the weight loader's expect_tx arrival
      mbar_init(wempty_bar(s), 1);  // the (pair's) MMA commit
    }
    for (int s = 0; s < KT; ++s) {
      mbar_init(tfull_bar(s), kTokThreads);  // one arrival per loader thread (cp.async, or the TMA expect_tx)
      mbar_init(tempty_bar(s), 1);
      mbar_init(pfull_bar(s), 1);  // pair: the MMA thread's expect_tx; the partner's relay brings the bytes
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(afull_bar(a), 1);
      // a pair's accumulators live in both CTAs: both epilogues release them
      mbar_init(aempty_bar(a), PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    // claimed ids are read by the MMA thread, 4 token-loader warps and the
    // epilogue warps, and in a pair also by the second CTA's weight loader;
    // the pair's first CTA claims for both
    const uint32_t n_id = PAIR ? 2 * (1 + 4 + kEpiWarps) + 1 : 1 + 4 + kEpiWarps;
    for (int r = 0; r < kRing; ++r) {
      mbar_init(id_full(r), 1);
      mbar_init(id_empty(r), n_id);
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
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), L::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the partner's barriers exist before anything reaches them
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
        local += on ? chunk_count<BN, PAIR>(seg_count(p, seg_off, s)) * seg_nrb<PAIR>(p, ph, s == p.E) : 0;
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      int run = incl - local;
      for (int s = s0; s < min(nseg, s0 + per); ++s) {
        ts[s] = run;
        run += on ? chunk_count<BN, PAIR>(seg_count(p, seg_off, s)) * seg_nrb<PAIR>(p, ph, s == p.E) : 0;
      }
      if (lane == 31) ts[nseg] = incl;
    }
  }
  __syncthreads();
  const int total = start1[nseg] + start2[nseg];
  unsigned *err = p.err;
  unsigned *claim = p.sync + kSyncClaim;
  unsigned *done1 = p.sync + kSyncDone;  // gate/up tiles finished, per segment (one count per CTA of a tile)
  bool ok = true;

  // claimed ids: wait for one / hand its slot back (to the claiming CTA)
  auto wait_id = [&](int r, uint32_t parity) -> bool {
    if constexpr (PAIR) return mbar_wait_cluster(id_full(r), parity, err, abort_flag);
    else return mbar_wait(id_full(r), parity, err, abort_flag);
  };
  auto release_id = [&](int r) {
    if constexpr (PAIR) {
      if (rank != 0) {
        mbar_arrive_cluster(map_cluster(id_empty(r), 0));
        return;
      }
    }
    mbar_arrive(id_empty(r));
  };

  if (warp == kWWarp) {
    // ================= claims (first CTA) and weight loads (one thread)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      int ws = 0;
      uint32_t wph = 0;
      uint32_t issued = 0, issued_par = 0;  // per weight slot: a load issued, and its phase parity
      for (int i = 0; ok; ++i) {
        const int r = i % kRing;
        const uint32_t rph = (uint32_t)(i / kRing) & 1u;
        int t;
        if (rank == 0) {
          ok = mbar_wait(id_empty(r), rph ^ 1u, err, abort_flag);
          if (!ok) break;
          const int t0 = (int)atomicAdd(claim, 1u);
          t = t0 < total ? t0 : -1;
          ring[r] = t;
          if constexpr (PAIR) {
            st_cluster_u32(map_cluster(smem_u32(const_cast<int *>(ring + r)), 1), (uint32_t)t);
            mbar_arrive_cluster(map_cluster(id_full(r), 1));
          }
          mbar_arrive(id_full(r));
        } else {
          ok = wait_id(r, rph);
          if (!ok) break;
          t = ring[r];
          release_id(r);
        }
        if (t < 0) break;
        const Tile tl = decode_tile<BN, PAIR>(p, t, start1, start2, seg_off, nseg);
        // this CTA's 128 rows of each weight block of the tile
        const int i0 = tl.rb * tile_rows<PAIR>(tl.phase) + rank * 128;
        const int i1 = i0 + tile_rows<PAIR>(tl.phase) / 2;  // down: the second block
        for (int kb = 0; kb < tl.nk; ++kb) {
          ok = mbar_wait(wempty_bar(ws), wph ^ 1u, err, abort_flag);
          if (!ok) break;
          const int k0 = kb * 64;
          mbar_arrive_expect_tx(wfull_bar(ws), (uint32_t)kABytes);
          issued |= 1u << ws;
          issued_par = (issued_par & ~(1u << ws)) | (wph << ws);
          const uint32_t a0 = w_smem(ws), a1 = a0 + 16384;
          if (tl.phase == 0) {
            if (tl.shared) {
              tma_load_2d_hint(a0, &p.map_sg, wfull_bar(ws), k0, i0, pol_w);
              tma_load_2d_hint(a1, &p.map_su, wfull_bar(ws), k0, i0, pol_w);
            } else {
              tma_load_3d_hint(a0, &p.map_wg, wfull_bar(ws), k0, i0, tl.seg, pol_w);
              tma_load_3d_hint(a1, &p.map_wu, wfull_bar(ws), k0, i0, tl.seg, pol_w);
            }
          } else {
            if (tl.shared) {
              tma_load_2d_hint(a0, &p.map_sd, wfull_bar(ws), k0, i0, pol_w);
              tma_load_2d_hint(a1, &p.map_sd, wfull_bar(ws), k0, i1, pol_w);
            } else {
              tma_load_3d_hint(a0, &p.map_wd, wfull_bar(ws), k0, i0, tl.seg, pol_w);
              tma_load_3d_hint(a1, &p.map_wd, wfull_bar(ws), k0, i1, tl.seg, pol_w);
            }
          }
          if (++ws == KW) {
            ws = 0;
            wph ^= 1u;
          }
        }
      }
      if (!ok)
        for (int s = 0; s < KW; ++s)
          if ((issued >> s) & 1u) mbar_wait_drain(wfull_bar(s), (issued_par >> s) & 1u);
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
      ok = __all_sync(0xffffffffu, wait_id(r, (uint32_t)(i / kRing) & 1u));
      if (!ok) break;
      const int t = ring[r];
      __syncwarp();
      if (lane == 0) release_id(r);
      if (t < 0) break;
      const Tile tl = decode_tile<BN, PAIR>(p, t, start1, start2, seg_off, nseg);
      // this CTA's token rows of the chunk: all N, or in a pair its half
      const int tok_n = PAIR ? tl.N >> 1 : tl.N;
      const int tok_lo = rank * tok_n;

      // ---- a down tile needs every gate/up tile of its segment
      if (tl.phase == 1 && (p.phases & 1) && tid == 0) {
        const unsigned need = (unsigned)(chunk_count<BN, PAIR>(seg_count(p, seg_off, tl.seg)) *
                                         seg_nrb<PAIR>(p, 0, tl.shared) * (PAIR ? 2 : 1));
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
      const __nv_bfloat16 *src[L::kTokRows / 16];
      if (tl.phase == 0) {
        bool bad = false;
#pragma unroll
        for (int j = 0; j < L::kTokRows / 16; ++j) {
          const int row = rbase + 16 * j;
          const int cr = tok_lo + row;  // row within the chunk
          const int rr = cr < tl.ntok ? cr : 0;
          int tok = 0;
          if (row < tok_n) {
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
          for (int j = 0; j < L::kTokRows / 16; ++j) {
            const int row = rbase + 16 * j;
            if (row < tok_n) cp_async_16(bs + row * 128 + ((c8 ^ (row & 7)) << 4), src[j] + k0);
          }
          cp_async_arrive_noinc(tfull_bar(ts));
        } else if (tid == 0) {
          // activation rows row0 + tok_lo + [0, tok_n) (contiguous, tok_n a
          // multiple of 16): boxes of 128 rows while they fit, then 64/32/16
          mbar_arrive_expect_tx(tfull_bar(ts), (uint32_t)(tok_n * 128));
          issued |= 1u << ts;
          issued_par = (issued_par & ~(1u << ts)) | (tph << ts);
          const CUtensorMap *mb = tl.shared ? p.map_acts : p.map_act;
          int off = 0;
          while (tok_n - off >= 128) {
            tma_load_2d(bs + (uint32_t)off * 128, &mb[3], tfull_bar(ts), k0, tl.row0 + tok_lo + off);
            off += 128;
          }
#pragma unroll
          for (int bi = 2; bi >= 0; --bi) {
            const int h = 16 << bi;
            if (tok_n - off >= h) {
              tma_load_2d(bs + (uint32_t)off * 128, &mb[bi], tfull_bar(ts), k0, tl.row0 + tok_lo + off);
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
    if (lane == 0 && rank == 0) {
      // ================= MMA issuer (a pair's first CTA issues for both)
      int ws = 0, ts = 0;
      uint32_t wph = 0, tph = 0;
      bool any = false;
      for (int i = 0; ok; ++i) {
        const int r = i % kRing;
        ok = wait_id(r, (uint32_t)(i / kRing) & 1u);
        if (!ok) break;
        const int t = ring[r];
        release_id(r);
        if (t < 0) break;
        const Tile tl = decode_tile<BN, PAIR>(p, t, start1, start2, seg_off, nseg);
        const int acc = i % L::kAccBufs;
        const uint32_t aph = (uint32_t)(i / L::kAccBufs) & 1u;
        ok = mbar_wait(aempty_bar(acc), aph ^ 1u, err, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)(acc * 2 * BN);
        const uint32_t d1 = d0 + (uint32_t)BN;
        const uint32_t idesc = idesc_bf16(PAIR ? 256 : 128, tl.N);
        for (int kb = 0; kb < tl.nk; ++kb) {
          ok = mbar_wait(wfull_bar(ws), wph, err, abort_flag) && mbar_wait(tfull_bar(ts), tph, err, abort_flag);
          if (PAIR && ok) {  // the partner's slots of this K step (its relay signals 4 bytes)
            mbar_arrive_expect_tx(pfull_bar(ts), 4u);
            ok = mbar_wait_cluster(pfull_bar(ts), tph, err, abort_flag);
          }
          if (!ok) break;
          if (tl.phase == 0) fence_proxy_async_smem();  // token rows were written by cp.async
          tc_fence_after();
          const uint64_t a0 = sdesc_sw128(w_smem(ws));
          const uint64_t a1 = sdesc_sw128(w_smem(ws) + 16384);
          const uint64_t bd = sdesc_sw128(t_smem(ts));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            if constexpr (PAIR) {
              umma_bf16_pair(d0, a0 + 2 * kk, bd + 2 * kk, idesc, accum);
              umma_bf16_pair(d1, a1 + 2 * kk, bd + 2 * kk, idesc, accum);
            } else {
              umma_bf16(d0, a0 + 2 * kk, bd + 2 * kk, idesc, accum);
              umma_bf16(d1, a1 + 2 * kk, bd + 2 * kk, idesc, accum);
            }
          }
          any = true;
          if constexpr (PAIR) {  // release the slots of both CTAs
            umma_commit_pair_mc(wempty_bar(ws), kBoth);
            umma_commit_pair_mc(tempty_bar(ts), kBoth);
          } else {
            umma_commit(wempty_bar(ws));
            umma_commit(tempty_bar(ts));
          }
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
        if constexpr (PAIR) umma_commit_pair_mc(afull_bar(acc), kBoth);
        else umma_commit(afull_bar(acc));
      }
      if (!ok && any) {
        if constexpr (PAIR) umma_commit_pair_mc(drain_bar, 1);
        else umma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0);
      }
    } else if (PAIR && lane == 0) {
      // ================= the pair's second CTA: relay "my slots of K step q
      // are full" to the first CTA's MMA thread
      int ws = 0, ts = 0;
      uint32_t wph = 0, tph = 0;
      for (int i = 0; ok; ++i) {
        const int r = i % kRing;
        ok = wait_id(r, (uint32_t)(i / kRing) & 1u);
        if (!ok) break;
        const int t = ring[r];
        release_id(r);
        if (t < 0) break;
        const Tile tl = decode_tile<BN, PAIR>(p, t, start1, start2, seg_off, nseg);
        for (int kb = 0; kb < tl.nk; ++kb) {
          ok = mbar_wait(wfull_bar(ws), wph, err, abort_flag) && mbar_wait(tfull_bar(ts), tph, err, abort_flag);
          if (!ok) break;
          fence_proxy_async_smem();  // token rows written by cp.async, read by the partner's MMAs
          st_async_signal(map_cluster(smem_u32(relay_word + ts), 0), (uint32_t)kb, map_cluster(pfull_bar(ts), 0));
          if (++ws == KW) {
            ws = 0;
            wph ^= 1u;
          }
          if (++ts == KT) {
            ts = 0;
            tph ^= 1u;
          }
        }
      }
    }
  } else {
    // ================= epilogue (warps 6..13 -> TMEM lane quarters 2,3,0,1, twice)
    const int q = warp & 3;
    // column groups of kEpiCols (32 for wide tiles: one TMEM wait per 32 columns);
    // the lane quarter's warps take groups in turn
    constexpr int kEpiCols = BN >= 64 ? kWideEpiCols : 16;
    constexpr int kEpiStep = kEpiCols * (kEpiWarps / 4);
    const int c_first = kEpiCols * ((warp - kEpiWarp0) >> 2);
    __nv_bfloat16 *stage = reinterpret_cast<__nv_bfloat16 *>(smem + L::kEpiOff + (warp - kEpiWarp0) * kEpiCols * 64);
    const int r = 32 * q + lane;  // TMEM lane = this CTA's weight row within a 128-row block
    for (int i = 0; ok; ++i) {
      const int rs = i % kRing;
      ok = __all_sync(0xffffffffu, wait_id(rs, (uint32_t)(i / kRing) & 1u));
      if (!ok) break;
      const int t = ring[rs];
      __syncwarp();
      if (lane == 0) release_id(rs);
      if (t < 0) break;
      const Tile tl = decode_tile<BN, PAIR>(p, t, start1, start2, seg_off, nseg);
      const int acc = i % L::kAccBufs;
      const uint32_t aph = (uint32_t)(i / L::kAccBufs) & 1u;
      ok = __all_sync(0xffffffffu, mbar_wait(afull_bar(acc), aph, err, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint32_t t0 = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * 2 * BN);
      // first weight row of this CTA's D0 / D1 blocks
      const int row_a = tl.rb * tile_rows<PAIR>(tl.phase) + rank * 128;
      const int row_b = row_a + tile_rows<PAIR>(tl.phase) / 2;
      if constexpr (L::kStageEpi) {
        // lane j of the warp owns weight row first + j; a group of ncol tokens is
        // written to the staging block as [token][32 rows] bf16, then each lane
        // stores 16 bytes (8 rows of one token): 4 lanes per token row piece
        auto flush = [&](__nv_bfloat16 *rows, size_t ld, int first, int limit, int c, int ncol) {
          __syncwarp();
          for (int pass = 0; pass < ncol / 8; ++pass) {
            const int jj = pass * 8 + (lane >> 2), qq = lane & 3;
            const uint4 v = *reinterpret_cast<const uint4 *>(stage + jj * 32 + qq * 8);
            if (c + jj < tl.ntok && first + qq * 8 < limit)
              *reinterpret_cast<uint4 *>(rows + (size_t)(c + jj) * ld + first + qq * 8) = v;
          }
          __syncwarp();
        };
        if (tl.phase == 0) {
          const int ld = tl.shared ? p.Is : p.I;
          __nv_bfloat16 *rows = (tl.shared ? p.act_s : p.act) + (size_t)tl.row0 * ld;
          const int first = row_a + 32 * q;
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
            flush(rows, (size_t)ld, first, ld, c, ncol);
          }
        } else {
          __nv_bfloat16 *rows = (tl.shared ? p.y_s : p.y) + (size_t)tl.row0 * p.H;
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
            flush(rows, (size_t)p.H, row_a + 32 * q, p.H, c, ncol);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < ncol) stage[j * 32 + lane] = __float2bfloat16_rn(vb[j]);
            flush(rows, (size_t)p.H, row_b + 32 * q, p.H, c, ncol);
          }
        }
      } else if (tl.phase == 0) {
        const int ld = tl.shared ? p.Is : p.I;
        __nv_bfloat16 *out = tl.shared ? p.act_s : p.act;
        const int ii = row_a + r;
        for (int c = c_first; c < tl.N; c += kEpiStep) {
          for (int c16 = c; c16 < min(c + kEpiCols, tl.N); c16 += 16) {
            float g[16], u[16];
            tmem_ld16(t0 + (uint32_t)c16, g);
            tmem_ld16(t0 + (uint32_t)(BN + c16), u);
            tmem_wait_ld();
            if (ii < ld) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c16 + j < tl.ntok)
                  out[(size_t)(tl.row0 + c16 + j) * ld + ii] = __float2bfloat16_rn(silu_mul(g[j], u[j]));
            }
          }
        }
      } else {
        __nv_bfloat16 *out = tl.shared ? p.y_s : p.y;
        const int ha = row_a + r, hb = row_b + r;
        for (int c = c_first; c < tl.N; c += kEpiStep) {
          for (int c16 = c; c16 < min(c + kEpiCols, tl.N); c16 += 16) {
            float va[16], vb[16];
            tmem_ld16(t0 + (uint32_t)c16, va);
            tmem_ld16(t0 + (uint32_t)(BN + c16), vb);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (c16 + j < tl.ntok) {
                __nv_bfloat16 *row = out + (size_t)(tl.row0 + c16 + j) * p.H;
                if (ha < p.H) row[ha] = __float2bfloat16_rn(va[j]);
                if (hb < p.H) row[hb] = __float2bfloat16_rn(vb[j]);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // release the accumulator (a pair's live in both CTAs; its MMA thread is in the first)
        if (PAIR && rank != 0) mbar_arrive_cluster(map_cluster(aempty_bar(acc), 0));
        else mbar_arrive(aempty_bar(acc));
      }
      if (tl.phase == 0 && (p.phases & 2)) {
        // publish: this CTA's share of the gate/up tile is written (release to the down tiles)
        __threadfence();
        named_bar_sync(2, 32 * kEpiWarps);
        if (warp == kEpiWarp0 && lane == 0) atomicAdd(done1 + tl.seg, 1u);
      }
    }
  }

  __syncwarp();
  __syncthreads();
  // a pair frees its TMEM together, and neither CTA leaves while the other may
  // still signal its barriers
  if constexpr (PAIR) cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, L::kTmemCols);
    else tmem_dealloc(tmem, L::kTmemCols);
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

int gemm_tile_n(int T) {
  if (T <= 16) return 16;
  if (T <= 32) return 32;
  if (T <= 64) return 64;
  if (T <= 128) return 128;
  return 256;
}

namespace {
template <int BN, bool PAIR>
cudaError_t launch_one(const GemmParams &p, int num_ctas, cudaStream_t stream, bool pdl) {
  using L = Layout<BN, PAIR>;
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(expert_ffn_kernel<BN, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::kSmem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  void *args[] = {(void *)&p};
  const int ctas = PAIR ? num_ctas & ~1 : num_ctas;
  return launch_ex((const void *)expert_ffn_kernel<BN, PAIR>, dim3(ctas), dim3(kGemmThreads), L::kSmem, stream, pdl,
                   PAIR ? 2 : 1, args);
}
}  // namespace

// 256-token tiles run on CTA pairs (clusters of two, 2-SM MMA); the narrow
// tiles of small batches run one CTA per tile.
cudaError_t launch_expert_ffn(const GemmParams &p, int bn, int num_ctas, cudaStream_t stream, bool pdl) {
  switch (bn) {
    case 16: return launch_one<16, false>(p, num_ctas, stream, pdl);
    case 32: return launch_one<32, false>(p, num_ctas, stream, pdl);
    case 64: return launch_one<64, false>(p, num_ctas, stream, pdl);
    case 128: return launch_one<128, false>(p, num_ctas, stream, pdl);
    case 256: return num_ctas >= 2 ? launch_one<256, true>(p, num_ctas, stream, pdl)
                                   : launch_one<256, false>(p, num_ctas, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
