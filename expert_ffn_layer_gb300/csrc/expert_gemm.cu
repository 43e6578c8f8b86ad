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
// Scheduling.  CTAs (one per SM) claim tiles from an atomic counter in a fixed
// order (see "Claim order" below): an early block of shared-expert gate/up
// tiles, the remaining gate/up tiles, then every down tile.  A down tile is
// thus claimed only after every gate/up tile has been claimed by a running
// CTA: its wait for the gate/up tiles of its segment (a per-segment completion
// count, bounded) can always be satisfied, whatever the residency of other
// CTAs.  Gate/up tiles never wait.  In the layer chain the early block needs
// no routing, so it runs while the router and the permutation still do
// (programmatic dependent launch: the routing kernels let this one launch as
// soon as they start).  The last CTA to leave zeroes the counters for the next
// call.
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
// Warp roles: 0 claims tiles and issues the weight TMA loads (lane 0) and
// builds the claim-order tables once the routing is visible (whole warp); 1-4
// load token rows (cp.async) or activation rows (TMA, one thread) and wait for
// a down tile's gate/up tiles; 5 and 22 issue the MMAs of the first and second
// accumulator of the pair (one thread each; 5 owns TMEM);
// 6-21 drain the accumulators, four warps per TMEM lane quarter taking its
// 16-column groups in turn (the epilogue of a wide tile is not overlapped with
// MMAs, so the more warps drain it the sooner TMEM is free: sixteen warps beat
// eight by 2-3 % on the wide tiles).  For BN <= 128 two TMEM accumulator pairs overlap one
// tile's epilogue with the next tile's MMAs (BN = 256 fills TMEM with one pair).
#include <cuda_fp8.h>

#include "fp8.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "silu.cuh"

namespace moe {

namespace {

constexpr int kABytes = 2 * 128 * 128;  // weights of one K step: two 128-row x 64-bf16 boxes
constexpr int kMaxSeg = 258;            // E <= 256 routed + 1 shared (+1 sentinel)
// Gate/up runs of the claim order (the down phase's order has a closed form):
// at most 1 + 256 (grouped level-major) or E + 2 (segment-major).
constexpr int kMaxRuns = 260;
// Shared-expert gate/up tiles claimed ahead of everything else (whole row-block
// levels, at least one): in the layer chain they run before the routing is known.
constexpr int kEarlyTiles = 32;
constexpr int kGroupSegs = 32;  // routed segments per group of the level-major gate/up order
constexpr int kWWarp = 0;               // tile claims + weight loads (lane 0)
constexpr int kTokWarp0 = 1;            // warps 1-4: token / activation loads
constexpr int kTokThreads = 128;
constexpr int kMmaWarp = 5;             // issues the first accumulator's MMAs, owns TMEM
constexpr int kEpiWarp0 = 6;            // warps 6.. : the epilogue
constexpr int kEpiWarps = 16;
constexpr int kMma2Warp = kEpiWarp0 + kEpiWarps;  // issues the second accumulator's MMAs
constexpr int kGemmThreads = 32 * (kMma2Warp + 1);
constexpr int kWideEpiCols = 16;        // epilogue column group of tiles of 64 tokens or more
constexpr int kRing = 4;                // claimed tile ids in flight
// FP8 weights: TMA brings the E4M3 codes of a K step (two 128-row x 64-code
// boxes, 16 KB) into a ring of their own; eight converter warps (taking the
// place of eight epilogue warps) write them as bf16 into the weight slots
constexpr int kQBytes = 2 * 128 * 64;
constexpr int kCvtWarps = 8;
constexpr unsigned long long kDrainNs = 20000000ull;
// Kernel modes: bf16 weights; FP8 weights expanded to bf16 in shared memory by
// converter warps (weight-only); W8A8 -- FP8 weights and FP8 activations fed
// straight to kind::f8f6f4 MMAs (K steps of 128 codes: 128-byte rows again).
constexpr int kModeBF16 = 0, kModeQ8 = 1, kModeF8 = 2;

// Ring depths: weight slots of 32 KB and token slots of BN x 128 bytes; with
// FP8 weights, code slots of 16 KB (the bytes in flight from HBM) and three
// bf16 weight slots between the converters and the MMAs.
template <int BN, int MODE>
struct Rings {
  static constexpr bool Q8 = MODE == kModeQ8;
  static constexpr int kW = Q8 ? 3 : BN >= 256 ? 3 : BN >= 240 ? 4 : BN >= 128 ? 5 : 6;
  static constexpr int kQ = Q8 ? (BN >= 128 ? 4 : 6) : 0;
  static constexpr int kT = BN >= 64 ? 3 : 4;
};

template <int BN, int MODE>
struct Layout {
  static constexpr bool Q8 = MODE == kModeQ8;
  static constexpr int kW = Rings<BN, MODE>::kW;
  static constexpr int kQ = Rings<BN, MODE>::kQ;
  static constexpr int kT = Rings<BN, MODE>::kT;
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
  static constexpr int kNumBars = 2 * kW + 2 * kT + 6 + 2 * kRing + 2 * kQ;
  // tmem slot, abort flag, ring of tile ids, schedule scalars (SchedMisc),
  // then the decoded tiles of the ring (kRing x 32 bytes)
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
  static constexpr int kTilesOff = kMiscOff + 128;
  static constexpr int kSegOffOff = kTilesOff + 32 * kRing;   // routed segment offsets [E + 1]
  static constexpr int kCstOff = kSegOffOff + 4 * kMaxSeg;    // routed chunk prefix [E + 1]
  static constexpr int kRunStartOff = kCstOff + 4 * kMaxSeg;  // first tile of each run [runs + 1]
  static constexpr int kRunDescOff = kRunStartOff + 4 * (kMaxRuns + 1);
  static constexpr int kBytes = kRunDescOff + 4 * kMaxRuns;
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
  static_assert(MODE != kModeF8 || BN <= 240, "the W8A8 epilogue has no staged (256-token) form");
};

struct Tile {
  int phase;  // 0 gate/up, 1 down, 2 W8A8 activation quantisation of one chunk
  int seg, rb, row0, ntok, N, nk, shared;
};
static_assert(sizeof(Tile) == 32, "a ring entry of the decoded tiles");

// W8A8 quantisation tiles per chunk row: one tile per 256 activation columns
// when chunks are wide and experts average at most 256 tokens (the work of a
// chunk then spreads over several SMs; Hy3 prefill 1.49 -> 1.13 ms), else one
// per chunk (short chunks at decode, many chunks per expert on larger batches,
// where the extra tiles cost more than they balance).
template <int BN>
__device__ __forceinline__ int quant_blocks(const GemmParams &p, int ld) {
  return (BN >= 128 && p.S <= 256 * p.E) ? (ld + 255) >> 8 : 1;
}

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

// Claim order.  Tiles are numbered in the order CTAs claim them, as runs:
//   early block  the shared expert's gate/up tiles of row blocks [0, r_e) --
//                 they need only `hidden`, so in the layer chain they start
//                 before the routing is known (no table needed to decode them);
//   gate/up      grouped level-major (gu_order 1): the routed segments in groups
//                 (about 32 each), group after group; inside a group, for each
//                 128-row block r, a "level" run of every segment's chunks at r;
//                 after each group, its share of the shared expert's remaining
//                 row blocks.  In-flight tiles then mix experts of every size --
//                 few-token tiles that stream weights from HBM and many-token
//                 chunks whose weights are L2 hits -- so the two bounds overlap
//                 across SMs, while a group's experts still finish early enough
//                 for their down tiles not to wait.  Or segment-major (gu_order 0): each
//                 routed segment's row blocks in turn (chunks innermost), then the
//                 shared expert's remaining row blocks, which keeps one expert's
//                 token rows hot in L2 across its row blocks (many-token batches);
//   down         each routed segment's row blocks in turn (chunks innermost: the
//                 activations of a chunk are re-read from L2 by its row blocks),
//                 with the shared expert's row blocks spread evenly between
//                 them instead of forming one long compute-bound run.
// A run is either one segment's row blocks [rb, rb + cnt) in (row block,
// chunk) order, or a level (all routed segments of one group at one row block).
constexpr int kRunLevel = 1 << 30;
__host__ __device__ constexpr int run_desc(int seg, int rb, int cnt) { return seg | (rb << 9) | (cnt << 17); }
__device__ __forceinline__ int run_seg(int d) { return d & 0x1FF; }
__device__ __forceinline__ int run_rb(int d) { return (d >> 9) & 0xFF; }

// Scalars of the claim order that depend only on the dims (known before routing).
struct Sched {
  int nch_s;    // chunks of the shared segment (T tokens)
  int Rr, Rs;   // gate/up row blocks of a routed / the shared expert (0 when not run)
  int Rd;       // down row blocks (0 when not run)
  int r_e;      // shared row blocks in the early block
  int n_early;  // r_e * nch_s
  int ngroups, gsize;  // grouped level-major gate/up order: groups of gsize routed segments
};
template <int BN>
__device__ __forceinline__ Sched make_sched(const GemmParams &p) {
  Sched q;
  const bool gu = p.phases & 1, dn = p.phases & 2, sh = p.has_shared != 0;
  q.nch_s = sh ? chunk_count<BN>(p.T) : 0;
  q.Rr = gu ? (p.I + 127) >> 7 : 0;
  q.Rs = (gu && sh) ? (p.Is + 127) >> 7 : 0;
  q.Rd = dn ? (p.H + 255) >> 8 : 0;
  q.r_e = q.Rs > 0 ? max(1, min(q.Rs, kEarlyTiles / q.nch_s)) : 0;
  q.n_early = q.r_e * q.nch_s;
  // groups of about kGroupSegs segments, few enough that their level runs fit
  // the run table (at most 256 + 8 gate/up runs)
  q.ngroups = max(1, min((p.E + kGroupSegs - 1) / kGroupSegs, 256 / (q.Rr + 1)));
  q.gsize = (p.E + q.ngroups - 1) / q.ngroups;
  return q;
}

// Tables written once per CTA (by warp 0, after the routing is visible) and
// read by every role: schedule totals in shared memory.
struct SchedMisc {
  int total;      // tiles of all phases
  int n_gu_runs;  // gate/up runs (their tiles end at G1)
  int G1;         // first tile after the gate/up tiles (W8A8: the first quantisation tile)
  int GD;         // first down tile (G1 unless W8A8)
};

template <int BN, int KSH>
__device__ __forceinline__ Tile decode_tile(const GemmParams &p, int t, const Sched &q, const SchedMisc &m,
                                            const int *seg_off, const int *cst, const int *rstart, const int *rdesc) {
  Tile tl;
  int seg, rb, ch;
  bool quant = false;
  if (t < q.n_early) {
    tl.phase = 0;
    seg = p.E;
    rb = t / q.nch_s;
    ch = t - rb * q.nch_s;
  } else if (t < m.G1) {
    tl.phase = 0;
    int lo = 0, hi = m.n_gu_runs;  // the last run starting at or before t (rstart[n_gu_runs] = G1)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (rstart[mid] <= t) lo = mid;
      else hi = mid;
    }
    const int d = rdesc[lo];
    const int local = t - rstart[lo];
    if (d & kRunLevel) {
      rb = run_rb(d);
      const int s_lo = run_seg(d) * q.gsize;  // the group's segments [s_lo, s_hi)
      const int key = local + cst[s_lo];
      int a = s_lo, b = min(p.E, s_lo + q.gsize);  // the last segment whose chunks start at or before key
      while (b - a > 1) {
        const int mid = (a + b) >> 1;
        if (cst[mid] <= key) a = mid;
        else b = mid;
      }
      seg = a;
      ch = key - cst[a];
    } else {
      seg = run_seg(d);
      const int nch = seg == p.E ? q.nch_s : cst[seg + 1] - cst[seg];
      const int qq = local / nch;
      rb = run_rb(d) + qq;
      ch = local - qq * nch;
    }
  } else if (t < m.GD) {
    // W8A8: one quantisation tile per chunk, routed segments in order, then the
    // shared expert's chunks
    tl.phase = 2;
    quant = true;
    const int u = t - m.G1, C = cst[p.E], Qr = quant_blocks<BN>(p, p.I), Qs = quant_blocks<BN>(p, p.Is);
    if (u < C * Qr) {
      const int cu = u / Qr;
      rb = u - cu * Qr;  // the tile's block of activation columns
      int a = 0, b = p.E;  // the last segment whose chunks start at or before cu
      while (b - a > 1) {
        const int mid = (a + b) >> 1;
        if (cst[mid] <= cu) a = mid;
        else b = mid;
      }
      seg = a;
      ch = cu - cst[a];
    } else {
      seg = p.E;
      const int v = u - C * Qr;
      ch = v / Qs;
      rb = v - ch * Qs;
    }
  } else {
    // down: routed segment s starts at Rd cst[s] + nsh(s) nch_s, with nsh(s) =
    // floor(s nsd / E) shared row blocks placed before it; those placed after it
    // follow its own tiles
    tl.phase = 1;
    const int u = t - m.GD;
    const int nsd = p.has_shared ? q.Rd : 0;
    auto dstart = [&](int x) { return q.Rd * cst[x] + (x * nsd / p.E) * q.nch_s; };
    int a = 0, b = p.E;  // dstart(E) = every down tile > u
    while (b - a > 1) {
      const int mid = (a + b) >> 1;
      if (dstart(mid) <= u) a = mid;
      else b = mid;
    }
    const int nch = cst[a + 1] - cst[a];
    const int end = dstart(a) + q.Rd * nch;
    if (u < end) {
      seg = a;
      const int local = u - dstart(a);
      rb = local / nch;
      ch = local - rb * nch;
    } else {
      seg = p.E;
      const int v = u - end;
      rb = a * nsd / p.E + v / q.nch_s;
      ch = v - (v / q.nch_s) * q.nch_s;
    }
  }
  tl.seg = seg;
  tl.shared = seg == p.E ? 1 : 0;
  tl.rb = rb;
  const int cnt = tl.shared ? p.T : seg_off[seg + 1] - seg_off[seg];
  const int base = chunk_base<BN>(cnt);
  const int pin = ch * base;
  tl.ntok = min(base, cnt - pin);
  tl.row0 = (tl.shared ? 0 : seg_off[seg]) + pin;
  tl.N = (tl.ntok + 15) & ~15;
  tl.nk = quant ? 0 : tl.phase == 0 ? (p.H >> KSH) : ((tl.shared ? p.Is : p.I) >> KSH);  // K steps of 2^KSH
  return tl;
}

// Warp 0 builds the run tables once the routing (offsets) is visible.  Every
// lane fills its own entries; no entry depends on another lane's but through
// the chunk prefix, which the warp scans first.
template <int BN>
__device__ void build_sched_tables(const GemmParams &p, const Sched &q, SchedMisc *m, int *seg_off, int *cst,
                                   int *rstart, int *rdesc, int lane) {
  const int E = p.E;
  for (int i = lane; i <= E; i += 32) seg_off[i] = __ldg(p.offsets + i);
  __syncwarp();
  bool good = true;
  for (int i = lane; i <= E; i += 32) {
    if (i == 0) good = good && seg_off[0] == 0;
    else good = good && seg_off[i] >= seg_off[i - 1];
    if (i == E) good = good && seg_off[i] == p.S;
  }
  good = __all_sync(0xffffffffu, good);
  if (!good && blockIdx.x == 0 && lane == 0 && p.err != nullptr) atomicOr(p.err, MOE_DEVERR_OFFSETS);
  // routed chunk prefix (no routed work at all when the offsets are bad)
  const int per = (E + 31) / 32, s0 = lane * per, s1 = min(E, s0 + per);
  int local = 0;
  for (int s = s0; s < s1; ++s) local += good ? chunk_count<BN>(seg_off[s + 1] - seg_off[s]) : 0;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - local;
  for (int s = s0; s < s1; ++s) {
    cst[s] = run;
    run += good ? chunk_count<BN>(seg_off[s + 1] - seg_off[s]) : 0;
  }
  if (lane == 31) cst[E] = incl;
  __syncwarp();
  const int C = cst[E];
  // ---- gate/up runs
  const int base = q.Rs > 0 ? 1 : 0;  // run 0: the early block
  if (lane == 0 && base) {
    rstart[0] = 0;
    rdesc[0] = run_desc(E, 0, q.r_e);
  }
  int n_gu = base, G1 = q.n_early;
  if (p.gu_order == 1 && q.Rr > 0) {  // grouped level-major
    // lane g < ngroups: group g's level runs, then its share of the shared
    // expert's remaining row blocks; run and tile offsets by a scan over groups
    const int g = lane;
    const bool has = g < q.ngroups;
    const int s_lo = has ? min(E, g * q.gsize) : E, s_hi = has ? min(E, s_lo + q.gsize) : E;
    const int Cg = cst[s_hi] - cst[s_lo];
    const int rrem = max(0, q.Rs - q.r_e);
    const int lo_g = has ? g * rrem / q.ngroups : 0, hi_g = has ? (g + 1) * rrem / q.ngroups : 0;
    const int my_tiles = has ? q.Rr * Cg + (hi_g - lo_g) * q.nch_s : 0;
    const int my_runs = has ? q.Rr + (hi_g > lo_g ? 1 : 0) : 0;
    int t_incl = my_tiles, r_incl = my_runs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, t_incl, o), b = __shfl_up_sync(0xffffffffu, r_incl, o);
      if (lane >= o) {
        t_incl += a;
        r_incl += b;
      }
    }
    if (has) {
      int idx = base + r_incl - my_runs;
      const int st = q.n_early + t_incl - my_tiles;
      for (int r = 0; r < q.Rr; ++r, ++idx) {
        rstart[idx] = st + r * Cg;
        rdesc[idx] = kRunLevel | run_desc(g, r, 0);
      }
      if (hi_g > lo_g) {
        rstart[idx] = st + q.Rr * Cg;
        rdesc[idx] = run_desc(E, q.r_e + lo_g, hi_g - lo_g);
      }
    }
    n_gu += __shfl_sync(0xffffffffu, r_incl, 31);
  } else if (q.Rr > 0) {  // segment-major
    for (int s = lane; s < E; s += 32) {
      rstart[base + s] = q.n_early + q.Rr * cst[s];
      rdesc[base + s] = run_desc(s, 0, q.Rr);
    }
    n_gu += E;
    if (q.Rs > q.r_e) {
      if (lane == 0) {
        rstart[n_gu] = q.n_early + q.Rr * C;
        rdesc[n_gu] = run_desc(E, q.r_e, q.Rs - q.r_e);
      }
      ++n_gu;
    }
  }
  G1 += q.Rr * C + max(0, q.Rs - q.r_e) * q.nch_s;
  // ---- W8A8: a quantisation tile per chunk between the gate/up and the down tiles
  const int GD = G1 + (p.mode == 2 && q.Rd > 0 ? C * quant_blocks<BN>(p, p.I) +
                                                       (p.has_shared ? q.nch_s * quant_blocks<BN>(p, p.Is) : 0)
                                                 : 0);
  // ---- down tiles: routed segments in order, the shared row blocks spread
  // between them (closed form, see decode_tile)
  int total = GD;
  if (q.Rd > 0) total += q.Rd * C + (p.has_shared ? q.Rd : 0) * q.nch_s;
  if (lane == 0) {
    rstart[n_gu] = G1;
    m->total = total;
    m->n_gu_runs = n_gu;
    m->G1 = G1;
    m->GD = GD;
  }
  __threadfence_block();  // every lane's entries before lane 0 releases them (id_full)
  __syncwarp();
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

// max(p[first], p[first + step], ...) over indices < n, eight independent
// loads per round (the maxima were written by other CTAs: loaded through L2)
__device__ __forceinline__ float strided_max(const float *p, int first, int step, int n) {
  float m[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int b = first; b < n; b += 8 * step) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (b + u * step < n) m[u] = fmaxf(m[u], __ldcg(p + b + u * step));
  }
  return fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
}

// Column maxima of a warp's 32 rows x 16 columns: m[j] is this lane's value of
// column j.  Four halving exchanges (8 + 4 + 2 + 1 shuffles) and a last pair
// leave in m[0] the maximum over all 32 lanes of the column returned, which
// lanes 2c and 2c + 1 share for c = 0..15.
__device__ __forceinline__ int col_max16(float (&m)[16], int lane) {
#pragma unroll
  for (int half = 8, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
    const bool upper = lane & bit;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = upper ? m[k] : m[half + k];
      const float keep = upper ? m[half + k] : m[k];
      m[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, bit));
    }
  }
  m[0] = fmaxf(m[0], __shfl_xor_sync(0xffffffffu, m[0], 1));
  return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
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

// W8A8 quantisation tile: the activation rows of one chunk (or one block of 256
// of their columns, see quant_blocks) to E4M3 codes, once
// (each down row block then loads the codes by TMA instead of quantising the
// rows again).  Row scale = max |row| / 448 from the per-32-column maxima the
// gate/up epilogue kept; the quotients as the row quantiser forms them.  The
// 128 loader threads: rows rbase + 16 j, the 8 threads of a row taking its
// 16-value pieces c8, c8 + 8, ...  Activations and maxima were written by other
// CTAs: read through L2.
template <int BN>
__device__ __forceinline__ void quantize_chunk_rows(const GemmParams &p, const Tile &tl, int rbase, int c8) {
  const int ld = tl.shared ? p.Is : p.I, nb = ld >> 5, npc = ld >> 4;
  const bool split = quant_blocks<BN>(p, ld) > 1;  // this tile covers 256 columns (16 pieces) of each row
  const int pc0 = split ? tl.rb * 16 : 0, pc1 = split ? min(pc0 + 16, npc) : npc;
  const float *am = tl.shared ? p.amax_s : p.amax;
  const __nv_bfloat16 *act = tl.shared ? p.act_s : p.act;
  uint8_t *codes = tl.shared ? p.aq_s : p.aq;
  float *scales = tl.shared ? p.asc_s : p.asc;
#pragma unroll 1
  for (int j = 0; j < BN / 16; ++j) {
    const int row = rbase + 16 * j;
    float m = row < tl.ntok ? strided_max(am + (size_t)(tl.row0 + row) * nb, c8, 8, nb) : 0.0f;
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    if (row >= tl.ntok) continue;
    const float sc = e4m3_row_scale(m), rs = __frcp_rn(sc);
    if (c8 == 0 && pc0 == 0) scales[tl.row0 + row] = sc;
    const uint4 *src = reinterpret_cast<const uint4 *>(act + (size_t)(tl.row0 + row) * ld);
    uint4 *dst = reinterpret_cast<uint4 *>(codes + (size_t)(tl.row0 + row) * ld);
    for (int pc = pc0 + c8; pc < pc1; pc += 8) {
      const uint4 v0 = __ldcg(src + 2 * pc), v1 = __ldcg(src + 2 * pc + 1);
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      float f[16];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        f[2 * e] = e4m3_quotient(__uint_as_float(w[e] << 16), sc, rs);
        f[2 * e + 1] = e4m3_quotient(__uint_as_float(w[e] & 0xFFFF0000u), sc, rs);
      }
      dst[pc] = make_uint4(e4m3_pack4(f[0], f[1], f[2], f[3]), e4m3_pack4(f[4], f[5], f[6], f[7]),
                           e4m3_pack4(f[8], f[9], f[10], f[11]), e4m3_pack4(f[12], f[13], f[14], f[15]));
    }
  }
}

}  // namespace

template <int BN, int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1) expert_ffn_kernel(const __grid_constant__ GemmParams p) {
  using L = Layout<BN, MODE>;
  constexpr bool Q8 = MODE == kModeQ8, F8 = MODE == kModeF8;
  constexpr int KE = F8 ? 128 : 64;  // K elements per step: one 128-byte row of a weight or token box
  constexpr int KSH = F8 ? 7 : 6;
  constexpr int KW = L::kW, KT = L::kT, KQ = L::kQ, EW = L::kEpiW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = (uint64_t *)(smem + L::kBarOff);
  uint32_t *tmem_slot = (uint32_t *)(smem + L::kMiscOff);
  volatile int *abort_flag = (volatile int *)(smem + L::kMiscOff + 4);
  volatile int *ring = (volatile int *)(smem + L::kMiscOff + 16);  // kRing claimed tile ids
  SchedMisc *misc = (SchedMisc *)(smem + L::kMiscOff + 32);
  Tile *tiles = (Tile *)(smem + L::kTilesOff);  // the claimed tiles, decoded once by the claiming warp
  int *seg_off = (int *)(smem + L::kSegOffOff);
  int *cst = (int *)(smem + L::kCstOff);
  int *rstart = (int *)(smem + L::kRunStartOff);
  int *rdesc = (int *)(smem + L::kRunDescOff);

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
  auto drain_bar2 = smem_u32(&bars[2 * KW + 2 * KT + 5 + 2 * kRing + 2 * KQ]);
  auto q_smem = [&](int s) { return smem_u32(smem + L::kQOff + s * kQBytes); };
  auto w_smem = [&](int s) { return smem_u32(smem + s * kABytes); };
  auto t_smem = [&](int s) { return smem_u32(smem + L::kTOff + s * L::kTokBytes); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < KW; ++s) {
      mbar_init(wfull_bar(s), Q8 ? kCvtWarps / 2 : 1);  // the weight loader's expect_tx arrival, or one converter group
      mbar_init(wempty_bar(s), 2);                  // both MMA issuers' commits
    }
    for (int s = 0; s < KQ; ++s) {
      mbar_init(qfull_bar(s), 1);           // the loader's expect_tx arrival
      mbar_init(qempty_bar(s), kCvtWarps / 2);  // one converter group done reading
    }
    for (int s = 0; s < KT; ++s) {
      mbar_init(tfull_bar(s), kTokThreads);  // one arrival per loader thread (cp.async, or the TMA expect_tx)
      mbar_init(tempty_bar(s), 2);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(afull_bar(a), 2);
      mbar_init(aempty_bar(a), EW);
    }
    mbar_init(drain_bar, 1);
    mbar_init(drain_bar2, 1);
    for (int r = 0; r < kRing; ++r) {
      mbar_init(id_full(r), 1);
      mbar_init(id_empty(r), 2 + 4 + EW + (Q8 ? kCvtWarps : 0));  // MMA issuers, token loaders, epilogue, converters
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

  // Dependents may launch now: every kernel of this library waits for its
  // predecessor's completion before it reads what that one wrote.
  pdl_launch_dependents();
  // Routing data (perm, offsets) comes from the previous kernel.  With p.early
  // the early block's tiles (the shared expert's first row blocks) proceed
  // before it is visible, and each role waits only when it first meets a tile
  // that needs it; otherwise every thread waits here.
  if (!p.early) pdl_wait();
  const Sched q = make_sched<BN>(p);
  if (p.early && q.Rs > 0 && warp == kWWarp && lane == 0) {
    // The shared expert's weights into L2 while the routing still runs: none
    // of its tiles depends on the routing, and the early block alone would
    // stream them from a few SMs.  Each CTA takes a strided share of the
    // 64 x 128 boxes of ws_gate, ws_up and ws_down.
    const int kx_gu = p.H / KE, n_gu = kx_gu * ((p.Is + 127) / 128);
    const int kx_d = p.Is / KE, n_d = kx_d * ((p.H + 127) / 128);
    for (int b = blockIdx.x; b < 2 * n_gu + n_d; b += gridDim.x) {
      if (b < 2 * n_gu) {
        const int bb = b < n_gu ? b : b - n_gu;
        tma_prefetch_l2_2d(b < n_gu ? &p.map_sg : &p.map_su, (bb % kx_gu) * KE, (bb / kx_gu) * 128);
      } else {
        const int bb = b - 2 * n_gu;
        tma_prefetch_l2_2d(&p.map_sd, (bb % kx_d) * KE, (bb / kx_d) * 128);
      }
    }
  }
  unsigned *err = p.err;
  unsigned *claim = p.sync + kSyncClaim;
  unsigned *done1 = p.sync + kSyncDone;   // gate/up tiles finished, per segment
  unsigned *done2 = p.sync + kSyncQuant;  // W8A8: quantisation tiles finished, per segment
  bool ok = true;
  auto decode = [&](int t) { return decode_tile<BN, KSH>(p, t, q, *misc, seg_off, cst, rstart, rdesc); };

  if (warp == kWWarp) {
    // ================= tile claims and weight loads.  Lane 0 claims tiles and
    // issues the weight TMA loads (FP8 weights to the code slots, bf16 weights
    // straight to the weight slots); the whole warp builds the claim-order
    // tables when the first tile past the early block is claimed.
    constexpr int NS = Q8 ? KQ : KW;
    // Weights stream with the evict-first L2 policy.  256-token tiles (experts
    // averaging more than 256 tokens) split an expert into several chunks whose
    // tiles read the same weight rows at about the same time: there every chunk
    // but the segment's last loads them evict-last, so the later chunks find
    // them in L2 (zipf layer: 0.8 GB less DRAM traffic).  At 240-token tiles,
    // where few experts have several chunks, keeping lines cost more than it saved.
    const uint64_t pol_first = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    int ws = 0;
    uint32_t wph = 0;
    uint32_t issued = 0, issued_par = 0;  // per weight slot: a load issued, and its phase parity
    bool tables = false;
    for (int i = 0; ok; ++i) {
      const int r = i % kRing;
      ok = __all_sync(0xffffffffu, mbar_wait(id_empty(r), ((uint32_t)(i / kRing) & 1u) ^ 1u, err, abort_flag));
      if (!ok) break;
      int t0 = 0;
      if (lane == 0) t0 = (int)atomicAdd(claim, 1u);
      t0 = __shfl_sync(0xffffffffu, t0, 0);
      if (t0 >= q.n_early && !tables) {
        if (p.early) pdl_wait();
        build_sched_tables<BN>(p, q, misc, seg_off, cst, rstart, rdesc, lane);
        tables = true;
      }
      const int t = t0 < q.n_early ? t0 : (t0 < misc->total ? t0 : -1);
      Tile tl;
      if (lane == 0) {
        // the tile is decoded here, once, and published with its id: the other
        // roles read the decoded entry instead of searching the run tables
        if (t >= 0) {
          tl = decode(t);
          tiles[r] = tl;
        }
        ring[r] = t;
        mbar_arrive(id_full(r));  // release: the tables and the entry are visible to the roles that take this id
      }
      if (t < 0) break;
      if (lane == 0) {
        const int i0 = tl.rb * (tl.phase == 0 ? 128 : 256);
        uint64_t pol_w = pol_first;
        if (BN >= 256) {  // the shared expert's chunks too (all T tokens, starting at row 0)
          const int seg0 = tl.shared ? 0 : seg_off[tl.seg], cnt = tl.shared ? p.T : seg_off[tl.seg + 1] - seg0;
          const int last_row0 = seg0 + (chunk_count<BN>(cnt) - 1) * chunk_base<BN>(cnt);
          if (tl.row0 < last_row0) pol_w = pol_keep;
        }
        for (int kb = 0; kb < tl.nk; ++kb) {
          const uint32_t fb = Q8 ? qfull_bar(ws) : wfull_bar(ws);
          ok = mbar_wait(Q8 ? qempty_bar(ws) : wempty_bar(ws), wph ^ 1u, err, abort_flag);
          if (!ok) break;
          const int k0 = kb * KE;
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
      ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
    }
    if (!ok && lane == 0)
      for (int s2 = 0; s2 < NS; ++s2)
        if ((issued >> s2) & 1u) mbar_wait_drain(Q8 ? qfull_bar(s2) : wfull_bar(s2), (issued_par >> s2) & 1u);
  } else if (warp < kTokWarp0 + 4) {
    // ================= token rows (gate/up) or activation rows (down)
    const int tid = threadIdx.x - 32 * kTokWarp0;  // 0..127
    const int c8 = tid & 7, rbase = tid >> 3;
    int ts = 0;
    uint32_t tph = 0;
    uint32_t issued = 0, issued_par = 0;  // per token slot: an activation TMA issued (thread 0)
    bool waited = !p.early;
    for (int i = 0; ok; ++i) {
      const int r = i % kRing;
      ok = __all_sync(0xffffffffu, mbar_wait(id_full(r), (uint32_t)(i / kRing) & 1u, err, abort_flag));
      if (!ok) break;
      const int t = ring[r];
      const Tile tl = tiles[r];
      __syncwarp();
      if (lane == 0) mbar_arrive(id_empty(r));
      if (t < 0) break;
      if (t >= q.n_early && !waited) {  // perm comes from the previous kernel
        pdl_wait();
        waited = true;
      }

      // ---- a down tile needs every gate/up tile of its segment -- with W8A8,
      // every quantisation tile of its segment, each of which needed those
      if (tl.phase >= 1 && (p.phases & 1) && tid == 0) {
        const int nch = tl.shared ? q.nch_s : cst[tl.seg + 1] - cst[tl.seg];
        const bool on_quant = F8 && tl.phase == 1;
        const unsigned *cnt = (on_quant ? done2 : done1) + tl.seg;
        const int nq = quant_blocks<BN>(p, tl.shared ? p.Is : p.I);  // quantisation tiles per chunk
        const unsigned need = (unsigned)(on_quant ? nch * nq : nch * (tl.shared ? q.Rs : q.Rr));
        if (ld_acquire_gpu(cnt) < need) {
          const unsigned long long t0 = globaltimer();
          while (ld_acquire_gpu(cnt) < need) {
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
      if constexpr (F8) {
        if (tl.phase == 2) {
          // W8A8 quantisation tile: every loader thread reads activations and
          // their row maxima itself, after thread 0's acquire of the count
          named_bar_sync(3, kTokThreads);
          quantize_chunk_rows<BN>(p, tl, rbase, c8);
          __threadfence();  // the codes and scales, before the count (release)
          named_bar_sync(3, kTokThreads);
          if (tid == 0) atomicAdd(done2 + tl.seg, 1u);
          continue;
        }
      }

      // ---- token rows of this thread for a gate/up tile: rows rbase + 16 j, as
      // 16-byte pieces of 128-byte K-step rows (64 bf16 values, or with W8A8 the
      // 128 E4M3 codes of the token's quantised row)
      const uint8_t *src[BN / 16];
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
          src[j] = F8 ? p.hq + (size_t)tok * p.H + c8 * 16
                      : reinterpret_cast<const uint8_t *>(p.hidden) + (size_t)tok * p.H * 2 + c8 * 16;
        }
        if (bad && err != nullptr) atomicOr(err, MOE_DEVERR_INDEX);
      }
      for (int kb = 0; kb < tl.nk; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(tempty_bar(ts), tph ^ 1u, err, abort_flag));
        if (!ok || *abort_flag) {
          ok = false;
          break;
        }
        const int k0 = kb * KE;
        const uint32_t bs = t_smem(ts);
        if (tl.phase == 0) {
#pragma unroll
          for (int j = 0; j < BN / 16; ++j) {
            const int row = rbase + 16 * j;
            if (row < tl.N) cp_async_16(bs + row * 128 + ((c8 ^ (row & 7)) << 4), src[j] + kb * 128);
          }
          cp_async_arrive_noinc(tfull_bar(ts));
        } else if (tid == 0) {
          // activation rows row0 .. row0 + N (contiguous, N a multiple of 16 and
          // <= 256; with W8A8 their E4M3 codes): boxes of 128 rows while they
          // fit, then one each of 64/32/16
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
  } else if (warp == kMmaWarp || warp == kMma2Warp) {
    // ================= MMA issuers: one thread per accumulator of the pair
    // (gate / up rows, or the two 128-row halves of w_down).  A tcgen05.mma
    // costs its issuing thread about 70 cycles whatever N is, so one thread
    // issuing both accumulators' four MMAs per K step (and two commits) could
    // not keep the tensor pipe busy below about N = 150; two threads issue in
    // parallel.  Each commits to the slot barriers (two arrivals free a slot).
    if (lane == 0) {
      const int half = warp == kMmaWarp ? 0 : 1;
      int ws = 0, ts = 0;
      uint32_t wph = 0, tph = 0;
      bool any = false;
      int na = 0;  // tiles that used an accumulator (quantisation tiles do not)
      for (int i = 0; ok; ++i) {
        const int r = i % kRing;
        ok = mbar_wait(id_full(r), (uint32_t)(i / kRing) & 1u, err, abort_flag);
        if (!ok) break;
        const int t = ring[r];
        const Tile tl = tiles[r];
        mbar_arrive(id_empty(r));
        if (t < 0) break;
        if (tl.phase == 2) continue;
        const int acc = na % L::kAccBufs;
        const uint32_t aph = (uint32_t)(na / L::kAccBufs) & 1u;
        ++na;
        ok = mbar_wait(aempty_bar(acc), aph ^ 1u, err, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t dh = tmem + (uint32_t)(acc * 2 * BN) + (uint32_t)(half * BN);
        const uint32_t idesc = F8 ? idesc_e4m3(128, tl.N) : idesc_bf16(128, tl.N);
        for (int kb = 0; kb < tl.nk; ++kb) {
          ok = mbar_wait(wfull_bar(ws), wph, err, abort_flag) && mbar_wait(tfull_bar(ts), tph, err, abort_flag);
          if (!ok) break;
          if (tl.phase == 0 || F8) fence_proxy_async_smem();  // token rows were written by cp.async / stores
          tc_fence_after();
          const uint64_t ah = sdesc_sw128(w_smem(ws) + (uint32_t)(half * 16384));
          const uint64_t bd = sdesc_sw128(t_smem(ts));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            if constexpr (F8) umma_f8(dh, ah + 2 * kk, bd + 2 * kk, idesc, accum);  // 32 codes of K per MMA
            else umma_bf16(dh, ah + 2 * kk, bd + 2 * kk, idesc, accum);
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
        const uint32_t db = half == 0 ? drain_bar : drain_bar2;
        umma_commit(db);
        mbar_wait_drain(db, 0);
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
    int na = 0;  // tiles that used an accumulator (quantisation tiles do not)
    for (int i = 0; ok; ++i) {
      const int rs = i % kRing;
      ok = __all_sync(0xffffffffu, mbar_wait(id_full(rs), (uint32_t)(i / kRing) & 1u, err, abort_flag));
      if (!ok) break;
      const int t = ring[rs];
      const Tile tl = tiles[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(id_empty(rs));
      if (t < 0) break;
      if (tl.phase == 2) continue;
      const int acc = na % L::kAccBufs;
      const uint32_t aph = (uint32_t)(na / L::kAccBufs) & 1u;
      ++na;
      ok = __all_sync(0xffffffffu, mbar_wait(afull_bar(acc), aph, err, abort_flag));
      if (!ok) break;
      tc_fence_after();
      if constexpr (F8) {  // a down tile's activation scales come from other CTAs' quantisation tiles
        if (tl.phase == 1 && (p.phases & 1)) (void)ld_acquire_gpu(done2 + tl.seg);
      }
      const uint32_t t0 = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * 2 * BN);
      // FP8 weights: the accumulators hold sum(value(code) * x); this lane's
      // row scales turn them into the products with the weights
      float s0 = 1.0f, s1 = 1.0f;
      if constexpr (Q8 || F8) {
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
              if constexpr (F8) {
                // W8A8: the accumulators hold code products; each row's weight scale
                // and each column's token scale make them gate and up.  The bf16
                // activation is stored, and its largest magnitude over this warp's
                // 32 rows is kept per column for the down tiles' quantisation.
                float cs = 0.0f;
                const int cj = c16 + (lane & 15);
                if (cj < tl.ntok) {
                  int tok = tl.shared ? tl.row0 + cj : __ldg(p.perm + tl.row0 + cj) / p.top_k;
                  tok = min(max(tok, 0), p.T - 1);
                  cs = __ldg(p.hs + tok);
                }
                float m[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  const float csj = __shfl_sync(0xffffffffu, cs, j);
                  m[j] = 0.0f;
                  if (c16 + j < tl.ntok && ii < ld) {
                    const __nv_bfloat16 b = __float2bfloat16_rn(silu_mul(g[j] * s0 * csj, u[j] * s1 * csj));
                    out[(size_t)(tl.row0 + c16 + j) * ld + ii] = b;
                    m[j] = fabsf(__bfloat162float(b));
                  }
                }
                const int col = col_max16(m, lane);  // lane's column of the warp-wide maxima (in m[0])
                if ((lane & 1) == 0 && c16 + col < tl.ntok)
                  (tl.shared ? p.amax_s : p.amax)[(size_t)(tl.row0 + c16 + col) * (ld >> 5) + tl.rb * 4 + q] = m[0];
              } else if (ii < ld) {
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
              float cs = 1.0f;
              if constexpr (F8) {
                // each column's activation scale, as its quantisation tile stored it
                const int cj = c16 + (lane & 15);
                if (cj < tl.ntok) cs = __ldcg((tl.shared ? p.asc_s : p.asc) + tl.row0 + cj);
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float csj = F8 ? __shfl_sync(0xffffffffu, cs, j) : 1.0f;
                if (c16 + j < tl.ntok) {
                  __nv_bfloat16 *row = out + (size_t)(tl.row0 + c16 + j) * p.H;
                  if (ha < p.H) __stcs(row + ha, __float2bfloat16_rn(Q8 ? va[j] * s0 : F8 ? va[j] * s0 * csj : va[j]));
                  if (hb < p.H) __stcs(row + hb, __float2bfloat16_rn(Q8 ? vb[j] * s1 : F8 ? vb[j] * s1 * csj : vb[j]));
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
    // Two groups of four converter warps take alternate K steps (the per-step
    // handoff -- waits, proxy fence, arrivals -- then overlaps across groups).
    // Warp wg of a group converts rows 64 (wg & 1) .. + 63 of box wg >> 1; per
    // pass, lane l converts 16 codes (chunk l & 3) of row 8 it + (l >> 2), so a
    // warp reads 512 contiguous bytes and writes whole 128-byte swizzled rows.
    // Parity waits stay unambiguous: with three weight slots a group's previous
    // step (j - 2) needed MMA j - 5 done, which orders the slot's earlier phase
    // (MMA j - 6) before its wait; with an even number of code slots, step
    // j - KQ belonged to the same group.
    static_assert(!Q8 || (KQ % 2 == 0 && KW == 3), "two converter groups need an even code ring and three weight slots");
    const int cw = warp - (kEpiWarp0 + EW);
    const int grp = cw >> 2, wg = cw & 3;
    const int box = wg >> 1, c = lane & 3;
    int ws = 0, qs = 0;
    uint32_t wph = 0, qph = 0;
    unsigned kstep = 0;
    for (int i = 0; ok; ++i) {
      const int rs = i % kRing;
      ok = __all_sync(0xffffffffu, mbar_wait(id_full(rs), (uint32_t)(i / kRing) & 1u, err, abort_flag));
      if (!ok) break;
      const int t = ring[rs];
      const Tile tl = tiles[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(id_empty(rs));
      if (t < 0) break;
      for (int kb = 0; kb < tl.nk; ++kb, ++kstep) {
        if ((int)(kstep & 1u) == grp) {
          ok = __all_sync(0xffffffffu, mbar_wait(qfull_bar(qs), qph, err, abort_flag) &&
                                           mbar_wait(wempty_bar(ws), wph ^ 1u, err, abort_flag));
          if (!ok) break;
          const uint8_t *src = smem + L::kQOff + qs * kQBytes + box * (kQBytes / 2);
          uint8_t *dst = smem + ws * kABytes + box * (kABytes / 2);
          uint4 v[8];  // every read first: the stores cannot then hold back the next loads
#pragma unroll
          for (int it = 0; it < 8; ++it)
            v[it] = *reinterpret_cast<const uint4 *>(src + (64 * (wg & 1) + 8 * it + (lane >> 2)) * 64 + c * 16);
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int rr = 64 * (wg & 1) + 8 * it + (lane >> 2);
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
      for (int i = 0; i < p.E + p.has_shared; ++i) s[kSyncDone + i] = 0;
      if (p.mode == kModeF8)
        for (int i = 0; i < p.E + p.has_shared; ++i) s[kSyncQuant + i] = 0;
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
template <int BN, int MODE>
cudaError_t launch_one(const GemmParams &p, int num_ctas, cudaStream_t stream, bool pdl) {
  using L = Layout<BN, MODE>;
  static thread_local unsigned long long attr_ctx = 0;
  const cudaError_t e = set_smem_attr_once((const void *)expert_ffn_kernel<BN, MODE>, (int)L::kSmem, attr_ctx);
  if (e != cudaSuccess) return e;
  void *args[] = {(void *)&p};
  return launch_ex((const void *)expert_ffn_kernel<BN, MODE>, dim3(num_ctas), dim3(kGemmThreads), L::kSmem, stream,
                   pdl, 1, args);
}
}  // namespace

cudaError_t launch_expert_ffn(const GemmParams &p, int bn, int num_ctas, cudaStream_t stream, bool pdl) {
  if (p.mode == kModeQ8) {  // weight-only FP8: narrow tiles only (the code ring takes the shared memory of wide token slots)
    switch (bn < 128 ? bn : 128) {
      case 16: return launch_one<16, kModeQ8>(p, num_ctas, stream, pdl);
      case 32: return launch_one<32, kModeQ8>(p, num_ctas, stream, pdl);
      case 64: return launch_one<64, kModeQ8>(p, num_ctas, stream, pdl);
      case 128: return launch_one<128, kModeQ8>(p, num_ctas, stream, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  if (p.mode == kModeF8) {  // W8A8: up to 240-token tiles (the epilogue has no staged form)
    switch (bn < 240 ? bn : 240) {
      case 16: return launch_one<16, kModeF8>(p, num_ctas, stream, pdl);
      case 32: return launch_one<32, kModeF8>(p, num_ctas, stream, pdl);
      case 64: return launch_one<64, kModeF8>(p, num_ctas, stream, pdl);
      case 128: return launch_one<128, kModeF8>(p, num_ctas, stream, pdl);
      case 240: return launch_one<240, kModeF8>(p, num_ctas, stream, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 16: return launch_one<16, kModeBF16>(p, num_ctas, stream, pdl);
    case 32: return launch_one<32, kModeBF16>(p, num_ctas, stream, pdl);
    case 64: return launch_one<64, kModeBF16>(p, num_ctas, stream, pdl);
    case 128: return launch_one<128, kModeBF16>(p, num_ctas, stream, pdl);
    case 240: return launch_one<240, kModeBF16>(p, num_ctas, stream, pdl);
    case 256: return launch_one<256, kModeBF16>(p, num_ctas, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
