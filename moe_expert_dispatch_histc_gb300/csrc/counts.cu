// counts.cu -- histc per logical rank, the logical all_gather, send/recv
// counts and the stable expert-major permutation ("NPU Training Operators -
// MC2", section "Execution path", steps 2-6).
//
// Three launches, no atomics on global memory and no floating point:
//   1. histc_warps:   each warp counts its sub-chunk of flat (token, slot)
//                     entries into a warp-private shared histogram over E+1
//                     bins (bin E = invalid id) and writes it to
//                     hist[bin * G + warp]  (bin-major, so the scan order
//                     (bin asc, warp asc) equals (expert asc, flat index asc)).
//   2. scan_counts:   one CTA: an exclusive scan of hist in that order ->
//                     base[bin * G + warp] = first permuted row of the warp's
//                     entries of that bin; offsets[e] = base[e * G]; per-rank
//                     counts cnt[W, E] and recv counts as differences of bases.
//   3. scatter_warps: each warp re-walks its sub-chunk 32 entries at a time;
//                     lanes with equal bins (match_bins) are ranked by
//                     a lane-mask popcount, giving a stable position.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace mc2 {

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Lanes whose bin equals this lane's (the mask __match_any_sync would give),
// from one ballot per bit of the bin: vote runs at a far higher rate than
// match, which made match the limit of a pass with few SMs.  Bins are 0..E;
// inactive lanes pass -1, whose low nbits bits (all ones) equal no bin since
// 2^nbits - 1 > E.
__device__ __forceinline__ uint32_t match_bins(int bin, int nbits) {
  uint32_t same = 0xffffffffu;
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (bin >> b) & 1;
    const uint32_t bal = __ballot_sync(0xffffffffu, bit);
    same &= bit ? bal : ~bal;
  }
  return same;
}

inline int match_bits(int E) {
  int n = 1;
  while ((1 << n) - 1 <= E) ++n;
  return n;
}

struct CountsParams {
  const int32_t* sel;
  int32_t* hist;
  int32_t* base;
  int32_t* cnt;
  int32_t* recv;
  int32_t* offsets;
  int32_t* permute_src;
  int32_t* unpermute_dst;
  int32_t* dev_status;
  int64_t RW, CPR, G;
  int E, W, EB, nbits;
};

__device__ __forceinline__ void warp_range(const CountsParams& p, int64_t g, int64_t& begin,
                                           int64_t& end) {
  const int64_t r = g / p.CPR, c = g % p.CPR;
  begin = r * p.RW + c * kCountsSub;
  end = begin + kCountsSub;
  const int64_t rank_end = (r + 1) * p.RW;
  if (end > rank_end) end = rank_end;
}

__global__ void __launch_bounds__(kCountsWarpsPerBlock * 32)
    histc_warps(CountsParams p) {
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kCountsWarpsPerBlock + warp;
  if (g >= p.G) return;
  int32_t* hist = sh + warp * p.EB;
  for (int b = lane; b < p.EB; b += 32) hist[b] = 0;
  __syncwarp();
  griddep_wait();
  griddep_launch_dependents();
  int64_t begin, end;
  warp_range(p, g, begin, end);
  bool bad = false;
  for (int64_t i0 = begin; i0 < end; i0 += 32) {
    const int64_t i = i0 + lane;
    const bool active = i < end;
    int bin = -1;
    if (active) {
      const int e = __ldg(p.sel + i);
      bin = (e >= 0 && e < p.E) ? e : p.E;
      bad |= (bin == p.E);
    }
    const uint32_t same = match_bins(bin, p.nbits);
    if (active && lane == __ffs(same) - 1) hist[bin] += __popc(same);
    __syncwarp();
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0 && p.dev_status) atomicOr(p.dev_status, 0x1);
  for (int b = lane; b < p.EB; b += 32) p.hist[static_cast<int64_t>(b) * p.G + g] = hist[b];
}

// Exclusive scan of one value per thread across the CTA (blockDim.x = 1024).
__device__ int64_t block_exclusive_scan(int64_t v, int64_t* warp_sums, int64_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t s = (lane < static_cast<int>(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive
  }
  __syncthreads();
  const int64_t warp_prefix = warp ? warp_sums[warp - 1] : 0;
  total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  return warp_prefix + x - v;
}

__global__ void __launch_bounds__(1024) scan_counts(CountsParams p) {
  __shared__ int64_t warp_sums[32];
  griddep_wait();
  griddep_launch_dependents();
  // exclusive scan of hist in (bin, warp) order; each thread scans a
  // contiguous segment, loading it with independent (unrolled) loads
  const int64_t N = static_cast<int64_t>(p.EB) * p.G;
  const int64_t seg = (N + blockDim.x - 1) / blockDim.x;
  const int64_t lo = threadIdx.x * seg;
  const int64_t hi = lo + seg < N ? lo + seg : N;
  int64_t own = 0;
#pragma unroll 8
  for (int64_t i = lo; i < hi; ++i) own += p.hist[i];
  int64_t total;
  int64_t run = block_exclusive_scan(own, warp_sums, total);
  for (int64_t i = lo; i < hi; ++i) {
    const int32_t v = p.hist[i];
    p.base[i] = static_cast<int32_t>(run);
    run += v;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= p.E; e += blockDim.x)
    p.offsets[e] = (p.G > 0) ? p.base[static_cast<int64_t>(e) * p.G] : 0;
  // per-rank histograms (the all_gather result) and recv counts: rank r's
  // warps are G-positions [r*CPR, (r+1)*CPR) of each bin, so its count of
  // expert e is the difference of two scan bases (the position after the
  // last warp of bin e is the first warp of bin e+1)
  const int El = p.E / p.W;
  for (int idx = threadIdx.x; idx < p.W * p.E; idx += blockDim.x) {
    const int r = idx / p.E, e = idx % p.E;
    const int64_t b0 = static_cast<int64_t>(e) * p.G + static_cast<int64_t>(r) * p.CPR;
    const int32_t c = (p.G > 0) ? p.base[b0 + p.CPR] - p.base[b0] : 0;
    p.cnt[idx] = c;
    // recv_counts of rank d = e / El: position (source r, local expert e % El)
    const int d = e / El, le = e % El;
    p.recv[static_cast<int64_t>(d) * p.W * El + r * El + le] = c;
  }
}

__global__ void __launch_bounds__(kCountsWarpsPerBlock * 32)
    scatter_warps(CountsParams p) {
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kCountsWarpsPerBlock + warp;
  if (g >= p.G) return;
  int32_t* run = sh + warp * p.EB;
  griddep_wait();
  griddep_launch_dependents();
  for (int b = lane; b < p.EB; b += 32) run[b] = p.base[static_cast<int64_t>(b) * p.G + g];
  __syncwarp();
  int64_t begin, end;
  warp_range(p, g, begin, end);
  const uint32_t lt = lanemask_lt();
  for (int64_t i0 = begin; i0 < end; i0 += 32) {
    const int64_t i = i0 + lane;
    const bool active = i < end;
    int bin = -1;
    if (active) {
      const int e = __ldg(p.sel + i);
      bin = (e >= 0 && e < p.E) ? e : p.E;
    }
    const uint32_t same = match_bins(bin, p.nbits);
    int32_t pos = 0;
    if (active) pos = run[bin] + __popc(same & lt);
    __syncwarp();
    if (active) {
      p.permute_src[pos] = static_cast<int32_t>(i);
      p.unpermute_dst[i] = pos;
      if (lane == __ffs(same) - 1) run[bin] += __popc(same);
    }
    __syncwarp();
  }
}

// ----------------------------------------------------------------------------
// Single-launch variant: one thread-block cluster of C CTAs (1024 threads
// each, C <= 16) runs all three steps, with the cluster's hardware barriers
// between them and the cross-CTA part of the scan read through distributed
// shared memory.  Same flat order, same chunking rule (chunks never straddle
// a rank), same stable positions as the three-launch pass -- only the chunk
// size differs, which changes no output.
//   chunk g (0 <= g < G = W*CPR) covers entries [r*RW + c*S, ...) of rank
//   r = g / CPR, c = g % CPR; CTA q owns chunks [q*GC, (q+1)*GC); its warp w
//   walks local chunks w, w+32, ...
// Shared memory per CTA: hist[EB][GC|1] (counts, then in place the first
// permuted row of each (bin, chunk)), cta_tot[EB], pre[EB], bin_start[EB+1].
// ----------------------------------------------------------------------------
struct ClusterCountsParams {
  const int32_t* sel;
  int32_t* cnt;
  int32_t* recv;
  int32_t* offsets;
  int32_t* permute_src;
  int32_t* unpermute_dst;
  int32_t* dev_status;
  int32_t* rank_base;  // global scratch [W, E]: first permuted row of rank r's entries of e
  int64_t RW;
  int CPR, S, G, GC, E, W, EB, nbits;
};

constexpr int kClusterCountsThreads = 1024;
constexpr int kClusterCountsMaxCtas = 16;

__device__ __forceinline__ void chunk_range(const ClusterCountsParams& p, int g, int64_t& begin,
                                            int64_t& end) {
  const int r = g / p.CPR, c = g - (g / p.CPR) * p.CPR;
  begin = static_cast<int64_t>(r) * p.RW + static_cast<int64_t>(c) * p.S;
  end = begin + p.S;
  const int64_t rank_end = static_cast<int64_t>(r + 1) * p.RW;
  if (end > rank_end) end = rank_end;
}

__global__ void __launch_bounds__(kClusterCountsThreads, 1)
    counts_cluster(ClusterCountsParams p) {
  extern __shared__ int32_t sh[];
  __shared__ int64_t warp_sums[32];
  const int EB = p.EB, GC = p.GC;
  const int GS = GC | 1;                    // odd row stride: no bank conflicts down a column
  int32_t* hist = sh;                       // [EB][GS]
  int32_t* cta_tot = hist + EB * GS;        // [EB]
  int32_t* pre = cta_tot + EB;              // [EB]
  int32_t* bin_start = pre + EB;            // [EB + 1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const uint32_t q = cluster_ctarank();
  const uint32_t nq = gridDim.x;            // one cluster: the grid
  const int g0 = static_cast<int>(q) * GC;

  for (int i = threadIdx.x; i < EB * GS; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();

  // 1. histc: warp-private columns of hist, 8 loads in flight per lane
  bool bad = false;
  for (int gl = warp; gl < GC && g0 + gl < p.G; gl += nwarps) {
    int64_t begin, end;
    chunk_range(p, g0 + gl, begin, end);
    for (int64_t i0 = begin; i0 < end; i0 += 256) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t i = i0 + u * 32 + lane;
        v[u] = i < end ? __ldg(p.sel + i) : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (i0 + u * 32 >= end) break;
        if (i0 + u * 32 + lane < end) {  // counts need no ranking: shared-memory atomics
          const int bin = (v[u] >= 0 && v[u] < p.E) ? v[u] : p.E;
          bad |= bin == p.E;
          atomicAdd(&hist[bin * GS + gl], 1);
        }
      }
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0 && p.dev_status) atomicOr(p.dev_status, 0x1);
  __syncthreads();
  // per-bin totals of this CTA's chunks: one warp per bin, lanes across chunks
  for (int b = warp; b < EB; b += nwarps) {
    int32_t t = 0;
    for (int gl = lane; gl < GC; gl += 32) t += hist[b * GS + gl];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) cta_tot[b] = t;
  }
  cluster_sync();

  // 2. scan in (bin, chunk) order across the cluster
  for (int b = threadIdx.x; b < EB; b += blockDim.x) {
    int32_t v[kClusterCountsMaxCtas];
#pragma unroll
    for (int r = 0; r < kClusterCountsMaxCtas; ++r)
      v[r] = r < static_cast<int>(nq)
                 ? static_cast<int32_t>(ld_shared_cluster_u32(map_to_rank(cta_tot + b, r)))
                 : 0;
    int32_t tot = 0, before = 0;
#pragma unroll
    for (int r = 0; r < kClusterCountsMaxCtas; ++r) {
      tot += v[r];
      if (r < static_cast<int>(q)) before += v[r];
    }
    bin_start[b] = tot;  // replaced by the exclusive scan below
    pre[b] = before;
  }
  __syncthreads();
  {
    const int seg = (EB + blockDim.x - 1) / blockDim.x;
    const int lo = threadIdx.x * seg, hi = min(lo + seg, EB);
    int64_t own = 0;
    for (int b = lo; b < hi; ++b) own += bin_start[b];
    int64_t total;
    int64_t run = block_exclusive_scan(own, warp_sums, total);
    for (int b = lo; b < hi; ++b) {
      const int32_t v = bin_start[b];
      bin_start[b] = static_cast<int32_t>(run);
      run += v;
    }
    if (threadIdx.x == 0) bin_start[EB] = static_cast<int32_t>(total);
  }
  __syncthreads();
  // first permuted row of each (bin, chunk): warp per bin, scan across lanes
  for (int b = warp; b < EB; b += nwarps) {
    int32_t run = bin_start[b] + pre[b];
    for (int gl0 = 0; gl0 < GC; gl0 += 32) {
      const int gl = gl0 + lane;
      const int32_t h = gl < GC ? hist[b * GS + gl] : 0;
      int32_t x = h;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (gl < GC) hist[b * GS + gl] = run + x - h;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  __syncthreads();
  if (q == 0)
    for (int e = threadIdx.x; e <= p.E; e += blockDim.x) p.offsets[e] = bin_start[e];
  // the first chunk of every rank lies in exactly one CTA
  for (int r = 0; r < p.W; ++r) {
    const int gl = r * p.CPR - g0;
    if (gl < 0 || gl >= GC) continue;
    for (int e = threadIdx.x; e < p.E; e += blockDim.x)
      p.rank_base[static_cast<int64_t>(r) * p.E + e] = hist[e * GS + gl];
  }
  cluster_sync();  // rank_base visible cluster-wide; no remote smem access after this

  // per-rank counts (the all_gather result) and recv counts
  const int El = p.E / p.W;
  for (int idx = static_cast<int>(q) * blockDim.x + threadIdx.x; idx < p.W * p.E;
       idx += nq * blockDim.x) {
    const int r = idx / p.E, e = idx - (idx / p.E) * p.E;
    const int32_t start = p.rank_base[idx];
    const int32_t stop = r + 1 < p.W ? p.rank_base[idx + p.E] : bin_start[e + 1];
    const int32_t c = stop - start;
    p.cnt[idx] = c;
    const int d = e / El, le = e - (e / El) * El;
    p.recv[static_cast<int64_t>(d) * p.W * El + r * El + le] = c;
  }

  // 3. stable scatter from each warp's running positions
  const uint32_t lt = lanemask_lt();
  for (int gl = warp; gl < GC && g0 + gl < p.G; gl += nwarps) {
    int64_t begin, end;
    chunk_range(p, g0 + gl, begin, end);
    for (int64_t i0 = begin; i0 < end; i0 += 256) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t i = i0 + u * 32 + lane;
        v[u] = i < end ? __ldg(p.sel + i) : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (i0 + u * 32 >= end) break;
        const int64_t i = i0 + u * 32 + lane;
        const bool active = i < end;
        int bin = -1;
        if (active) bin = (v[u] >= 0 && v[u] < p.E) ? v[u] : p.E;
        const uint32_t same = match_bins(bin, p.nbits);
        int32_t pos = 0;
        if (active) pos = hist[bin * GS + gl] + __popc(same & lt);
        __syncwarp();
        if (active) {
          p.permute_src[pos] = static_cast<int32_t>(i);
          p.unpermute_dst[i] = pos;
          if (lane == __ffs(same) - 1) hist[bin * GS + gl] += __popc(same);
        }
        __syncwarp();
      }
    }
  }
}

struct ClusterCountsPlan {
  int ctas = 0;   // 0: the plan does not fit; use the three-launch pass
  int CPR = 0, S = 0, G = 0, GC = 0;
  size_t smem = 0;
};

static ClusterCountsPlan plan_cluster_counts(const mc2_shape_t& s, int ctas) {
  ClusterCountsPlan pl;
  const int64_t R = static_cast<int64_t>(s.T) * s.k;
  const int64_t RW = R / s.W;
  if (R <= 0 || RW <= 0) return pl;
  // one chunk per warp when the ranks allow it
  const int64_t want = 32LL * ctas;
  int64_t cpr = std::max<int64_t>(1, (want + s.W - 1) / s.W);
  int64_t S = (RW + cpr - 1) / cpr;
  cpr = (RW + S - 1) / S;
  const int64_t G = cpr * s.W;
  const int64_t GC = (G + ctas - 1) / ctas;
  const int64_t EB = s.E + 1;
  const size_t smem = static_cast<size_t>(EB * (GC | 1) + 3 * EB + 1) * sizeof(int32_t);
  if (G > (1LL << 30) || smem > 160 * 1024) return pl;
  pl.ctas = ctas;
  pl.CPR = static_cast<int>(cpr);
  pl.S = static_cast<int>(S);
  pl.G = static_cast<int>(G);
  pl.GC = static_cast<int>(GC);
  pl.smem = smem;
  return pl;
}

// Cluster size for R entries: ~2K entries per CTA (each warp walks its chunk
// serially, so spreading over SMs shortens the pass), at most 16 CTAs, and no
// more than the GPU can co-schedule (checked once per size and device).
static int cluster_counts_ctas(int64_t R) {
  struct Fits { bool at[kClusterCountsMaxCtas + 1]; };
  static PerDevice<Fits> setup;
  const Fits fits = once_per_device(setup, [] {
    Fits r = {};
    cudaFuncSetAttribute(counts_cluster, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaFuncSetAttribute(counts_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
    for (int c = 1; c <= kClusterCountsMaxCtas; c *= 2) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(c);
      cfg.blockDim = dim3(kClusterCountsThreads);
      cfg.dynamicSmemBytes = 160 * 1024;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = c;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int n = 0;
      r.at[c] = cudaOccupancyMaxActiveClusters(&n, counts_cluster, &cfg) == cudaSuccess && n >= 1;
    }
    cudaGetLastError();  // clear anything the queries left
    return r;
  });
  int c = 1;
  while (c < kClusterCountsMaxCtas && static_cast<int64_t>(c) * 2048 < R) c *= 2;
  while (c > 1 && !fits.at[c]) c /= 2;
  return fits.at[c] ? c : 0;
}

static cudaError_t launch_counts_cluster(const mc2_shape_t& s, const ClusterCountsPlan& pl,
                                         const int32_t* sel, int32_t* cnt, int32_t* recv,
                                         int32_t* offsets, int32_t* permute_src,
                                         int32_t* unpermute_dst, int32_t* rank_base,
                                         int32_t* dev_status, cudaStream_t st) {
  ClusterCountsParams p;
  p.sel = sel;
  p.cnt = cnt;
  p.recv = recv;
  p.offsets = offsets;
  p.permute_src = permute_src;
  p.unpermute_dst = unpermute_dst;
  p.dev_status = dev_status;
  p.rank_base = rank_base;
  p.RW = static_cast<int64_t>(s.T) * s.k / s.W;
  p.CPR = pl.CPR;
  p.S = pl.S;
  p.G = pl.G;
  p.GC = pl.GC;
  p.E = s.E;
  p.W = s.W;
  p.EB = s.E + 1;
  p.nbits = match_bits(s.E);
  const cudaError_t e = launch_kernel(counts_cluster, dim3(pl.ctas), dim3(kClusterCountsThreads),
                                      pl.smem, st, pl.ctas, p);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

CountsGeom counts_geom(const mc2_shape_t& s) {
  CountsGeom g;
  g.R = static_cast<int64_t>(s.T) * s.k;
  g.RW = g.R / s.W;
  g.CPR = (g.RW + kCountsSub - 1) / kCountsSub;
  g.G = g.CPR * s.W;
  g.EB = s.E + 1;
  return g;
}

cudaError_t launch_counts(const mc2_shape_t& s, const int32_t* sel, int32_t* cnt, int32_t* recv,
                          int32_t* offsets, int32_t* permute_src, int32_t* unpermute_dst,
                          char* ws, int32_t* dev_status, cudaStream_t st) {
  const CountsGeom geo = counts_geom(s);
  const WsLayout L = ws_layout(s);
  const int path = counts_path_override();
  if (path != 1 && static_cast<int64_t>(s.T) * s.k > 0) {
    const int ctas = cluster_counts_ctas(static_cast<int64_t>(s.T) * s.k);
    const ClusterCountsPlan pl = ctas ? plan_cluster_counts(s, ctas) : ClusterCountsPlan{};
    if (pl.ctas)
      return launch_counts_cluster(s, pl, sel, cnt, recv, offsets, permute_src, unpermute_dst,
                                   reinterpret_cast<int32_t*>(ws + L.hist), dev_status, st);
  }
  CountsParams p;
  p.sel = sel;
  p.hist = reinterpret_cast<int32_t*>(ws + L.hist);
  p.base = reinterpret_cast<int32_t*>(ws + L.base);
  p.cnt = cnt;
  p.recv = recv;
  p.offsets = offsets;
  p.permute_src = permute_src;
  p.unpermute_dst = unpermute_dst;
  p.dev_status = dev_status;
  p.RW = geo.RW;
  p.CPR = geo.CPR;
  p.G = geo.G;
  p.E = s.E;
  p.W = s.W;
  p.EB = static_cast<int>(geo.EB);
  p.nbits = match_bits(s.E);
  const size_t smem = static_cast<size_t>(kCountsWarpsPerBlock) * geo.EB * sizeof(int32_t);
  const int blocks = static_cast<int>((geo.G + kCountsWarpsPerBlock - 1) / kCountsWarpsPerBlock);
  int launches = 0;
  cudaError_t err = cudaSuccess;
  if (blocks > 0) {
    err = launch_kernel(histc_warps, dim3(blocks), dim3(kCountsWarpsPerBlock * 32), smem, st, 1, p);
    if (err != cudaSuccess) return err;
    ++launches;
  }
  err = launch_kernel(scan_counts, dim3(1), dim3(1024), 0, st, 1, p);
  if (err != cudaSuccess) return err;
  ++launches;
  if (blocks > 0) {
    err = launch_kernel(scatter_warps, dim3(blocks), dim3(kCountsWarpsPerBlock * 32), smem, st, 1,
                        p);
    if (err != cudaSuccess) return err;
    ++launches;
  }
  note_launches(launches);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// Counts with library-owned scratch (mc2_moe_counts_static).
//
// Some callers cannot allocate device memory on their own: for example a
// plugin running inside a host application that owns every device
// allocation through its own pool, or a service whose device-memory budget
// is fixed when it starts.  For them the counts pass can use a fixed scratch
// array that lives in this library's device image instead of a caller
// workspace.  The array holds the two per-warp tables of the pass
// (histogram and scan base), kStaticCountsEntries int32 each (1 MiB in
// total); every GPU that loads the library keeps it until the process exits.
// The kernels write every entry they later read, so nothing in it needs
// clearing between calls.
// ----------------------------------------------------------------------------
constexpr int64_t kStaticCountsEntries = 131072;
constexpr int kStaticMaxDevices = 64;

static __device__ __align__(256) int32_t g_counts_scratch[2 * kStaticCountsEntries];

static std::mutex g_counts_scratch_mu;
static int32_t* g_counts_scratch_ptr[kStaticMaxDevices] = {};
static void* g_counts_scratch_ctx[kStaticMaxDevices] = {};

// The driver's cuCtxGetCurrent, looked up at run time (the library does not
// link the driver library).  Returns the current context, or NULL.
static void* current_context() {
  using Fn = int (*)(void**);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(ptr);
  });
  void* ctx = nullptr;
  if (fn && fn(&ctx) != 0) ctx = nullptr;
  return ctx;
}

// Device address of g_counts_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with that device current and cached per device, together with the
// context it was looked up in: after cudaDeviceReset (or any teardown of the
// primary context) the module is loaded again, possibly elsewhere, so a
// changed context triggers a fresh lookup instead of reusing a dangling
// address.
static cudaError_t counts_scratch_on_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kStaticMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_counts_scratch_mu);
  void* p = nullptr;
  if (!g_counts_scratch_ptr[dev]) {
    e = cudaGetSymbolAddress(&p, g_counts_scratch);   // also makes the context current
    if (e != cudaSuccess) return e;
    g_counts_scratch_ptr[dev] = static_cast<int32_t*>(p);
    g_counts_scratch_ctx[dev] = current_context();
  } else {
    void* ctx = current_context();
    if (ctx != g_counts_scratch_ctx[dev]) {
      e = cudaGetSymbolAddress(&p, g_counts_scratch);
      if (e != cudaSuccess) return e;
      g_counts_scratch_ptr[dev] = static_cast<int32_t*>(p);
      g_counts_scratch_ctx[dev] = current_context();
    }
  }
  *out = g_counts_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace mc2

extern "C" mc2_status_t mc2_moe_counts_static(const mc2_shape_t* s, const int32_t* sel,
                                              int32_t* cnt, int32_t* recv, int32_t* offsets,
                                              int32_t* permute_src, int32_t* unpermute_dst,
                                              int32_t* dev_status, void* stream) {
  using namespace mc2;
  reset_launches();
  if (mc2_check_shape(s) != MC2_OK) return MC2_ERR_INVALID_ARG;
  if (!cnt || !recv || !offsets) return MC2_ERR_INVALID_ARG;
  if (s->T > 0 && (!sel || !permute_src || !unpermute_dst)) return MC2_ERR_INVALID_ARG;
  if (!aligned({sel, cnt, recv, offsets, permute_src, unpermute_dst}))  // as mc2_moe_counts
    return MC2_ERR_INVALID_ARG;
  const CountsGeom geo = counts_geom(*s);
  if (geo.EB * geo.G > kStaticCountsEntries) return MC2_ERR_UNSUPPORTED;  // beyond the fixed scratch
  int32_t* scratch = nullptr;
  if (counts_scratch_on_current_device(&scratch) != cudaSuccess) return MC2_ERR_CUDA;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  CountsParams p;
  p.sel = sel;
  p.hist = scratch;
  p.base = scratch + kStaticCountsEntries;
  p.cnt = cnt;
  p.recv = recv;
  p.offsets = offsets;
  p.permute_src = permute_src;
  p.unpermute_dst = unpermute_dst;
  p.dev_status = dev_status;
  p.RW = geo.RW;
  p.CPR = geo.CPR;
  p.G = geo.G;
  p.E = s->E;
  p.W = s->W;
  p.EB = static_cast<int>(geo.EB);
  p.nbits = match_bits(s->E);
  const size_t smem = static_cast<size_t>(kCountsWarpsPerBlock) * geo.EB * sizeof(int32_t);
  const int blocks = static_cast<int>((geo.G + kCountsWarpsPerBlock - 1) / kCountsWarpsPerBlock);
  int launches = 0;
  if (blocks > 0) {
    histc_warps<<<blocks, kCountsWarpsPerBlock * 32, smem, st>>>(p);
    ++launches;
  }
  scan_counts<<<1, 1024, 0, st>>>(p);
  ++launches;
  if (blocks > 0) {
    scatter_warps<<<blocks, kCountsWarpsPerBlock * 32, smem, st>>>(p);
    ++launches;
  }
  note_launches(launches);
  return cudaGetLastError() == cudaSuccess ? MC2_OK : MC2_ERR_CUDA;
}
