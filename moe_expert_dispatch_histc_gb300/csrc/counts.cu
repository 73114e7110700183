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
//                     lanes with equal bins are ranked by __match_any_sync and
//                     a lane-mask popcount, giving a stable position.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace mc2 {

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
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
  int E, W, EB;
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
    const uint32_t same = __match_any_sync(0xffffffffu, bin);
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
    const uint32_t same = __match_any_sync(0xffffffffu, bin);
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

// Device address of g_counts_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
static cudaError_t counts_scratch_on_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kStaticMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_counts_scratch_mu);
  if (!g_counts_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_counts_scratch);
    if (e != cudaSuccess) return e;
    g_counts_scratch_ptr[dev] = static_cast<int32_t*>(p);
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
