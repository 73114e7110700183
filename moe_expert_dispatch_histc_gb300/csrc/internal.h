// internal.h -- declarations shared by the translation units of libmc2moe.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <initializer_list>
#include <mutex>

#include <utility>

#include "mc2moe.h"

namespace mc2 {

constexpr int kCountsSub = 256;       // flat (token, slot) entries per warp in the counts pass
constexpr int kCountsWarpsPerBlock = 8;
constexpr size_t kWsAlign = 256;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Pointer rule of the C ABI: every array 16-byte aligned (vector and TMA
// accesses), the workspace 256-byte aligned.  NULL passes (the null rules
// are separate).
inline bool aligned(std::initializer_list<const void*> ps, uintptr_t a = 16) {
  for (const void* p : ps)
    if (reinterpret_cast<uintptr_t>(p) & (a - 1)) return false;
  return true;
}

// Sub-chunk geometry of the counts pass: every logical rank's entries
// [r*RW, (r+1)*RW) are split into CPR chunks of kCountsSub (last one ragged),
// one warp each, so chunks never straddle ranks and G = W*CPR warps walk the
// flat order in sequence.
struct CountsGeom {
  int64_t R, RW, CPR, G, EB;  // EB = E + 1 bins (bin E collects invalid ids)
};
CountsGeom counts_geom(const mc2_shape_t& s);

// Grouped-GEMM modes.  MODE_FC1: fc1 + SwiGLU with the permute folded in
// (token rows gathered); MODE_FC2: fc2 -> scaled fp16 rows; MODE_FC1_ROWS:
// fc1 + SwiGLU on rows that are already permuted (the non-fused baseline
// path; plain TMA A tiles); MODE_FC1_PRE: fc1 with the permute folded in,
// writing the pre-activation gate|up rows G [R, 2I] in bf16 (the backward).
// MODE_FC2C: fc2 with the weighted combine fused in (the block's output is
// written by the fc2 kernel itself).
enum { MODE_FC1 = 0, MODE_FC2 = 1, MODE_FC1_ROWS = 2, MODE_FC1_PRE = 3, MODE_FC2C = 4 };

// Workspace layout (byte offsets from ws).
struct WsLayout {
  size_t hist, base;     // int32 [EB * G] each
  size_t y;              // fp16 [R, H] fc2 rows, expert-major, scaled (combine input)
  size_t yscale;         // fp32 [R, H/64] decode factor of each 64-column group of y
  size_t ctr;            // int32 [T, ceil(H/256)] row arrivals of the fused combine
  size_t defer;          // int32 count, then [T * ceil(H/256)] deferred (token, tile) sums
  size_t x_t32, w1_t32, w2_t32;  // fp32 tf32-rounded copies, weights transposed to [E, N, K] (act F32 only)
  size_t h_f32;          // fp32 [R, I] pre-requant SwiGLU output (act I8 only)
  size_t rowmax;         // uint32 [R] row absmax bits (act I8 only)
  size_t x_b16, hq_b16;  // bf16 copies of int8 operands (act I8 only)
  size_t w1_b16, w2_b16; // bf16 copies of int8 weights (act I8 only)
  size_t total;
};
WsLayout ws_layout(const mc2_shape_t& s);

uint64_t wait_limit_ns();
bool launch_overlap_enabled();  // programmatic dependent launch between the block's kernels
int counts_path_override();     // 0 auto, 1 three launches, 2 one cluster launch when it fits
int combine_path_override();    // 0 separate combine kernel, 1 fused into fc2 when supported
int mmrs_path_override();       // 0 fused (default), 1 two passes through int32 partials

// Launch `kernel` on `st` with programmatic stream serialization (so its
// prologue overlaps the previous kernel's tail; the kernel itself waits with
// griddepcontrol.wait before touching global memory) and, when cluster_x > 1,
// thread-block clusters of cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (launch_overlap_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
int tile_pairing_override();  // 0 auto, 1 single CTAs, 2 CTA pairs
void note_launches(int n);
void reset_launches();

// Launch wrappers (return cudaSuccess or the launch error).
cudaError_t launch_counts(const mc2_shape_t& s, const int32_t* sel, int32_t* cnt, int32_t* recv,
                          int32_t* offsets, int32_t* permute_src, int32_t* unpermute_dst,
                          char* ws, int32_t* dev_status, cudaStream_t st);

struct GemmArgs {
  const mc2_shape_t* s;
  const void* a;            // fc1: x [T, H]; fc2: h [R, I]
  const void* b;            // fc1: w1 [E, H, 2I]; fc2: w2 [E, I, H]
  const int32_t* offsets;
  const int32_t* permute_src;
  const float* a_scale;     // int8: per-token (fc1) or per-row (fc2)
  const float* b_scale;     // int8: per-channel
  void* out;                // fc1: h [R, I]; fc2: y [R, H] fp16 (scaled)
  float* yscale;            // fc2: [R, H/64]
  float* out_scale;         // unused by the GEMM itself
  uint32_t* rowmax;         // int8 fc1: row absmax bits
  int32_t* dev_status;
  int a_elem_bytes;         // 2 (bf16) or 4 (f32)
  int mode;                 // see gmm.cu
  // MODE_FC2C only: the combine's inputs and output
  const float* probs;
  const int32_t* unpermute_dst;
  int32_t* ctr;             // workspace counters [T, ceil(H/256)]
  int32_t* defer_items;     // workspace list [T * ceil(H/256)] of deferred sums
  int32_t* defer_count;     // workspace int32: its length
  void* comb_out;           // [T, H], bf16 (out_dtype MC2_BF16) or fp32
  int out_dtype;
};
cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t st);
// Whether the fc2 kernel can fuse the combine for this shape (top-k 1, 2, 4
// or 8); otherwise the separate combine kernel runs.
bool fused_combine_supported(const mc2_shape_t& s);
cudaError_t launch_permute_rows(const mc2_shape_t& s, const void* x, const int32_t* permute_src,
                                void* xp, cudaStream_t st);
// dW [E, M, N] fp32 = per expert A_e^T @ B_e over its permuted rows; A [R, M],
// B [R, N] bf16 (wgrad.cu).
cudaError_t launch_wgrad(const void* a, const void* b, const int32_t* offsets, int64_t R, int E,
                         int M, int N, float* dw, int32_t* dev_status, cudaStream_t st);

// int8 path (bf16 tensor cores holding int8 values, exact int32 sums)
struct QArgs {
  const mc2_shape_t* s;
  const void* a;            // fc1: x as bf16 [T, H]; fc2: h_q as bf16 [R, I]
  const void* b;            // bf16 copy of w1 [E, H, 2I] or w2 [E, I, H]
  const int32_t* offsets;
  const int32_t* permute_src;
  const float* a_scale;     // fc1: x scale [T]; fc2: h scale [R]
  const float* b_scale;     // fc1: w1 scale [E, 2I]; fc2: w2 scale [E, H]
  void* out;                // raw: int32 accumulators; else fc1 h fp32 [R, I], fc2 y fp16 [R, H]
  float* yscale;            // fc2 (not raw): [R, H/64]
  int32_t* dev_status;
  int mode;                 // 0 fc1, 1 fc2
  bool raw;
};
cudaError_t launch_gemm_q(const QArgs& g, cudaStream_t st);
cudaError_t launch_i8_to_bf16(const int8_t* src, void* dst, size_t n, cudaStream_t st);
// the same for two tensors in one launch
cudaError_t launch_i8_to_bf16_2(const int8_t* src0, void* dst0, size_t n0, const int8_t* src1,
                                void* dst1, size_t n1, cudaStream_t st);
cudaError_t launch_requant(const float* h, const int32_t* offsets, const mc2_shape_t& s, int8_t* hq,
                           float* hs, cudaStream_t st);

cudaError_t launch_combine(const mc2_shape_t& s, const void* y, const float* yscale,
                           const float* probs, const int32_t* offsets,
                           const int32_t* unpermute_dst, void* out, int out_dtype,
                           cudaStream_t st);
cudaError_t launch_round_tf32(const float* src, float* dst, size_t n, cudaStream_t st);
cudaError_t launch_transpose_round_tf32(const float* src, float* dst, int batch, int rows,
                                       int cols, cudaStream_t st);
cudaError_t launch_selftest_wait(uint64_t limit_ns, int32_t* dev_status, cudaStream_t st);

int num_sms();

// Host set-up that belongs to a device (kernel attributes, occupancy
// results): f() runs once for each device that is current at a call, and
// its result is kept per device, so a process that drives several GPUs sets
// each one up.
template <class T>
struct PerDevice {
  std::mutex m;
  uint64_t done = 0;
  T val[64] = {};
};

template <class T, class F>
T once_per_device(PerDevice<T>& o, F&& f) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return f();
  std::lock_guard<std::mutex> lk(o.m);
  if (!((o.done >> d) & 1u)) {
    o.val[d] = f();
    o.done |= uint64_t(1) << d;
  }
  return o.val[d];
}

// What a launcher needs to know once per device: whether the kernel accepted
// its shared-memory size, and (for kernels launched as CTA pairs) how many
// 2-CTA clusters of `threads` threads fit at once with `smem` bytes each.
struct KernelSetup {
  cudaError_t err;
  int pair_clusters;
};

template <typename... KArgs>
KernelSetup setup_kernel(void (*kernel)(KArgs...), size_t smem, int threads, bool pairs) {
  KernelSetup r{cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)),
                0};
  if (r.err != cudaSuccess || !pairs) return r;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms() & ~1), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&r.pair_clusters, kernel, &cfg) != cudaSuccess)
    r.pair_clusters = 0;
  return r;
}

}  // namespace mc2
