// Steps a3-a4: per-expert histogram, offsets and a stable permutation of the
// flat slots t*k + j into contiguous expert segments.
//
// "Hy3 Preview inference optimisation case", section 3 (FusedMoE, routing and
// index preprocessing): shared-memory block counts reserve one contiguous
// output range per expert.  The HunyuanImage 3.0 post (Routed Experts) fixes
// the slot numbering (flattened topk_idx) and the per-expert grouping.
//
// One CTA of 32 warps (8 for small batches).  Warp w owns a contiguous run of
// slots.  Pass 1 counts its run per expert in shared memory (warp match +
// popc); a column scan over
// the warps and a scan over the experts give every (warp, expert) pair its
// first output position; pass 2 walks the run again in slot order and ranks
// equal experts inside a warp with match/popc, so the order inside every
// segment is ascending slot order -- deterministic, no atomics on positions.
//
// Large batches (more than kPermuteOneCtaMax slots) run the same ranking on
// many CTAs.  The slots are cut into parts of kPartSlots.  A count kernel
// writes each part's per-expert count; the last part to finish turns the table
// into each part's first output position per expert (a prefix over the parts
// plus the expert offsets) and writes counts and offsets.  A scatter kernel
// then ranks each part's slots exactly as the one-CTA kernel does, starting
// from its row of the table, so both paths give the same permutation.
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {
constexpr int kMaxE = 256;
constexpr int kSmallS = 1024;  // up to this many slots the one-CTA kernel runs 8 warps
constexpr int kUnroll = 8;
}  // namespace

// One CTA of WARPS warps (32 for up to 8192 slots, 8 -- still one thread per
// expert in the column scan -- for up to 1024).
template <int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1) permute_kernel(const PermuteParams p) {
  constexpr int kWarps = WARPS, kThreads = WARPS * 32;
  static_assert(kThreads >= kMaxE, "one thread per expert in the column scan");
  __shared__ int base[kWarps][kMaxE];
  __shared__ int offs[kMaxE + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S, E = p.E;
  for (int i = threadIdx.x; i < kWarps * kMaxE; i += kThreads) (&base[0][0])[i] = 0;

  pdl_launch_dependents();  // dependents wait for this kernel's completion themselves
  pdl_wait();               // topk_idx comes from the router
  __syncthreads();

  const int chunk = (S + kWarps - 1) / kWarps;
  const int s_begin = min(S, warp * chunk), s_end = min(S, s_begin + chunk);
  bool bad = false;

  // pass 1: per-warp counts
  for (int s0 = s_begin; s0 < s_end; s0 += 32 * kUnroll) {
    int ev[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int s = s0 + 32 * u + lane;
      ev[u] = s < s_end ? __ldg(p.topk_idx + s) : 0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int s = s0 + 32 * u + lane;
      const bool valid = s < s_end;
      int e = ev[u];
      if (valid && (e < 0 || e >= E)) {
        bad = true;
        e = min(max(e, 0), E - 1);
      }
      const unsigned active = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const unsigned peers = __match_any_sync(active, e);
        if (lane == __ffs(peers) - 1) base[warp][e] += __popc(peers);
      }
    }
  }
  __syncthreads();

  // column scan over warps: base[w][e] <- sum_{w' < w} count[w'][e]; offs[e] <- total
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = base[w][e];
      base[w][e] = run;
      run += c;
    }
    offs[e] = run;
  }
  __syncthreads();

  // exclusive scan over experts (E <= 256 = 32 lanes x 8)
  if (warp == 0) {
    int vals[8], local = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      vals[j] = e < E ? offs[e] : 0;
      local += vals[j];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int excl = incl - local;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      if (e < E) {
        p.counts[e] = vals[j];
        offs[e] = excl;
      }
      excl += vals[j];
    }
    if (lane == 31) offs[E] = incl;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += kThreads) p.offsets[e] = offs[e];
  for (int i = threadIdx.x; i < kWarps * E; i += kThreads) {
    const int w = i / E, e = i - w * E;
    base[w][e] += offs[e];
  }
  __syncthreads();

  // pass 2: stable scatter in slot order
  for (int s0 = s_begin; s0 < s_end; s0 += 32 * kUnroll) {
    int ev[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int s = s0 + 32 * u + lane;
      ev[u] = s < s_end ? __ldg(p.topk_idx + s) : 0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int s = s0 + 32 * u + lane;
      const bool valid = s < s_end;
      const int e = min(max(ev[u], 0), E - 1);
      const unsigned active = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const unsigned peers = __match_any_sync(active, e);
        const int leader = __ffs(peers) - 1;
        int b = 0;
        if (lane == leader) {
          b = base[warp][e];
          base[warp][e] = b + __popc(peers);
        }
        b = __shfl_sync(active, b, leader);
        const int pos = b + __popc(peers & ((1u << lane) - 1u));
        p.perm[pos] = s;
        p.inv[s] = pos;
      }
    }
  }
  if (bad && p.err != nullptr) atomicOr(p.err, MOE_DEVERR_INDEX);
}

namespace {
constexpr int kPartThreads = 256;  // >= kMaxE: one thread per expert in the table pass
constexpr int kPartWarps = kPartThreads / 32;
constexpr int kWarpSlots = kPartSlots / kPartWarps;
static_assert(kPartThreads >= kMaxE, "one thread per expert");
static_assert(kWarpSlots % 32 == 0, "whole warp rounds");

// Exclusive prefix over the block's threads (kPartThreads); returns it and sets
// *total to the sum over all threads.
__device__ __forceinline__ int block_excl_scan(int v, int *warp_sums, int *total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kPartWarps; ++w) {
    const int x = warp_sums[w];
    before += w < warp ? x : 0;
    all += x;
  }
  *total = all;
  return before + incl - v;
}
}  // namespace

// Part g counts its slots per expert; the last part to finish builds the table.
__global__ void __launch_bounds__(kPartThreads) permute_count_kernel(const PermuteParams p) {
  __shared__ int cnt[kMaxE];
  __shared__ int warp_sums[kPartWarps];
  __shared__ int is_last;
  const int g = blockIdx.x, G = gridDim.x, E = p.E;
  for (int e = threadIdx.x; e < kMaxE; e += kPartThreads) cnt[e] = 0;

  pdl_launch_dependents();  // dependents wait for this kernel's completion themselves
  pdl_wait();               // topk_idx comes from the router
  __syncthreads();

  const int s0 = g * kPartSlots, s1 = min(p.S, s0 + kPartSlots);
  bool bad = false;
  for (int s = s0 + (int)threadIdx.x; s < s1; s += kPartThreads) {
    int e = __ldg(p.topk_idx + s);
    if (e < 0 || e >= E) {
      bad = true;
      e = min(max(e, 0), E - 1);
    }
    atomicAdd(&cnt[e], 1);
  }
  if (bad && p.err != nullptr) atomicOr(p.err, MOE_DEVERR_INDEX);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kPartThreads) p.part[(size_t)g * E + e] = cnt[e];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(p.done, 1u) == (unsigned)(G - 1) ? 1 : 0;
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // the last part: totals per expert, offsets, then each part's first position
  const int e = threadIdx.x;
  int tot = 0;
  if (e < E)
    for (int q = 0; q < G; ++q) tot += __ldcg(p.part + (size_t)q * E + e);
  int all = 0;
  const int first = block_excl_scan(e < E ? tot : 0, warp_sums, &all);
  if (e < E) {
    p.counts[e] = tot;
    p.offsets[e] = first;
    int run = first;
    for (int q = 0; q < G; ++q) {
      int *cell = p.part + (size_t)q * E + e;
      const int c = __ldcg(cell);
      *cell = run;
      run += c;
    }
  }
  if (threadIdx.x == 0) {
    p.offsets[E] = all;
    *p.done = 0;  // leave the header word zero for the next call
  }
}

// Part g ranks its slots: per-warp counts, a prefix over the part's warps from
// the part's row of the table, then the stable scatter (as the one-CTA kernel).
__global__ void __launch_bounds__(kPartThreads) permute_scatter_kernel(const PermuteParams p) {
  __shared__ int base[kPartWarps][kMaxE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x, E = p.E;
  for (int i = threadIdx.x; i < kPartWarps * kMaxE; i += kPartThreads) (&base[0][0])[i] = 0;

  pdl_launch_dependents();
  pdl_wait();  // the table and topk_idx come from the count kernel and the router
  __syncthreads();

  const int s0 = g * kPartSlots, s1 = min(p.S, s0 + kPartSlots);
  const int w0 = min(s1, s0 + warp * kWarpSlots), w1 = min(s1, w0 + kWarpSlots);
  constexpr int kRounds = kWarpSlots / 32;

  int ev[kRounds];
#pragma unroll
  for (int u = 0; u < kRounds; ++u) {
    const int s = w0 + 32 * u + lane;
    ev[u] = s < w1 ? min(max(__ldg(p.topk_idx + s), 0), E - 1) : 0;
  }
#pragma unroll
  for (int u = 0; u < kRounds; ++u) {
    const bool valid = w0 + 32 * u + lane < w1;
    const unsigned active = __ballot_sync(0xffffffffu, valid);
    if (valid) {
      const unsigned peers = __match_any_sync(active, ev[u]);
      if (lane == __ffs(peers) - 1) base[warp][ev[u]] += __popc(peers);
    }
  }
  __syncthreads();
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    int run = p.part[(size_t)g * E + e];
#pragma unroll
    for (int w = 0; w < kPartWarps; ++w) {
      const int c = base[w][e];
      base[w][e] = run;
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kRounds; ++u) {
    const int s = w0 + 32 * u + lane;
    const bool valid = s < w1;
    const unsigned active = __ballot_sync(0xffffffffu, valid);
    if (valid) {
      const int e = ev[u];
      const unsigned peers = __match_any_sync(active, e);
      const int leader = __ffs(peers) - 1;
      int b = 0;
      if (lane == leader) {
        b = base[warp][e];
        base[warp][e] = b + __popc(peers);
      }
      b = __shfl_sync(active, b, leader);
      const int pos = b + __popc(peers & ((1u << lane) - 1u));
      p.perm[pos] = s;
      p.inv[s] = pos;
    }
  }
}

cudaError_t launch_permute(const PermuteParams &p, cudaStream_t stream, bool pdl) {
  void *args[] = {(void *)&p};
  const int G = permute_parts(p.S);
  if (G == 0) {
    if (p.S <= kSmallS) return launch_ex((const void *)permute_kernel<8>, dim3(1), dim3(256), 0, stream, pdl, 1, args);
    return launch_ex((const void *)permute_kernel<32>, dim3(1), dim3(1024), 0, stream, pdl, 1, args);
  }
  cudaError_t e = launch_ex((const void *)permute_count_kernel, dim3(G), dim3(kPartThreads), 0, stream, pdl, 1, args);
  if (e != cudaSuccess) return e;
  return launch_ex((const void *)permute_scatter_kernel, dim3(G), dim3(kPartThreads), 0, stream, pdl, 1, args);
}

}  // namespace moe
