// mmrs.cu -- quantised matmul + reduce-scatter over W logical tensor-parallel
// ranks ("torch_npu.npu_mm_reduce_scatter_base", Ascend op-plugin docs,
// sections "Function description" and "Parameters"):
//
//   rank r holds x1_r [m, k] int8 with per-token scales x1_scale_r [m] and
//   x2_r [k, n] int8 with per-channel scales x2_scale_r [n];
//   out_r = rows [r*m/W, (r+1)*m/W) of  sum_r' (x1_scale_r' * x2_scale_r') *
//           (x1_r' @ x2_r')                              (reduce op: sum)
//
// On one GPU the W ranks are logical, so the reduce-scatter is a sum over the
// rank index and a row split.  Two passes:
//   1. the exact int8 grouped GEMM of the MoE block (gmm_q.cu, raw int32
//      accumulators; int8 values held as bf16, K summed in exact chunks) with
//      one group per rank: rows r*m .. r*m+m-1 of the stacked x1 against x2_r;
//   2. mmrs_reduce_kernel: per output element, the dequantised partials
//      (x1_scale * x2_scale) * float(acc) summed in fp32 in rank order, one
//      rounding to bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace mc2 {
namespace {

struct MmrsLayout {
  size_t x1_b16, x2_b16, acc, offsets, total;
};

bool mmrs_shape_ok(const mc2_mmrs_shape_t* s) {
  if (!s) return false;
  if (s->W < 1 || s->m < 0 || s->k < 64 || s->n < 64) return false;
  if (s->m % s->W || s->k % 64 || s->n % 64 || s->k > 4096) return false;
  const int64_t rows = static_cast<int64_t>(s->W) * s->m;
  return rows < (int64_t(1) << 31) && rows * s->n < (int64_t(1) << 40);
}

MmrsLayout mmrs_layout(const mc2_mmrs_shape_t& s) {
  MmrsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kWsAlign);
    return at;
  };
  const size_t rows = static_cast<size_t>(s.W) * s.m;
  L.x1_b16 = take(rows * s.k * 2);
  L.x2_b16 = take(static_cast<size_t>(s.W) * s.k * s.n * 2);
  L.acc = take(rows * s.n * 4);
  L.offsets = take(static_cast<size_t>(s.W + 1) * 4);
  L.total = off;
  return L;
}

__global__ void mmrs_offsets_kernel(int32_t* offsets, int W, int m) {
  griddep_wait();
  griddep_launch_dependents();
  for (int r = threadIdx.x; r <= W; r += blockDim.x) offsets[r] = r * m;
}

// out[i, c..c+7] = bf16( sum_r (xs[r, i] * ws[r, c]) * float(acc[r*m + i, c]) ), r ascending
__global__ void mmrs_reduce_kernel(const int32_t* __restrict__ acc, const float* __restrict__ xs,
                                   const float* __restrict__ ws, int W, int m, int n,
                                   __nv_bfloat16* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int n8 = n / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(m) * n8) return;
  const int64_t i = idx / n8;
  const int c = static_cast<int>(idx - i * n8) * 8;
  float s[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) s[j] = 0.f;
  for (int r = 0; r < W; ++r) {
    const float xr = __ldg(xs + static_cast<int64_t>(r) * m + i);
    const int4* a = reinterpret_cast<const int4*>(acc + (static_cast<int64_t>(r) * m + i) * n + c);
    const int4 a0 = __ldg(a), a1 = __ldg(a + 1);
    const float4* w = reinterpret_cast<const float4*>(ws + static_cast<int64_t>(r) * n + c);
    const float4 w0 = __ldg(w), w1 = __ldg(w + 1);
    s[0] += (xr * w0.x) * static_cast<float>(a0.x);
    s[1] += (xr * w0.y) * static_cast<float>(a0.y);
    s[2] += (xr * w0.z) * static_cast<float>(a0.z);
    s[3] += (xr * w0.w) * static_cast<float>(a0.w);
    s[4] += (xr * w1.x) * static_cast<float>(a1.x);
    s[5] += (xr * w1.y) * static_cast<float>(a1.y);
    s[6] += (xr * w1.z) * static_cast<float>(a1.z);
    s[7] += (xr * w1.w) * static_cast<float>(a1.w);
  }
  uint4 o;
  __nv_bfloat162 b;
  b = __floats2bfloat162_rn(s[0], s[1]);
  o.x = *reinterpret_cast<uint32_t*>(&b);
  b = __floats2bfloat162_rn(s[2], s[3]);
  o.y = *reinterpret_cast<uint32_t*>(&b);
  b = __floats2bfloat162_rn(s[4], s[5]);
  o.z = *reinterpret_cast<uint32_t*>(&b);
  b = __floats2bfloat162_rn(s[6], s[7]);
  o.w = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint4*>(out + i * n + c) = o;
}

bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace mc2

using namespace mc2;

extern "C" size_t mc2_mm_reduce_scatter_workspace_bytes(const mc2_mmrs_shape_t* s) {
  if (!mmrs_shape_ok(s)) return 0;
  const size_t t = mmrs_layout(*s).total;
  return t > kWsAlign ? t : kWsAlign;
}

extern "C" mc2_status_t mc2_mm_reduce_scatter_i8(const mc2_mmrs_shape_t* s, const int8_t* x1,
                                                 const float* x1_scale, const int8_t* x2,
                                                 const float* x2_scale, void* out, void* ws,
                                                 int32_t* dev_status, void* stream) {
  reset_launches();
  if (!mmrs_shape_ok(s)) return MC2_ERR_INVALID_ARG;
  if (!ws || !x2 || !x2_scale) return MC2_ERR_INVALID_ARG;
  if (s->m > 0 && (!x1 || !x1_scale || !out)) return MC2_ERR_INVALID_ARG;
  if (!al(x1, 16) || !al(x1_scale, 16) || !al(x2, 16) || !al(x2_scale, 16) || !al(out, 16) ||
      !al(ws, 256))
    return MC2_ERR_INVALID_ARG;
  if (s->m == 0) return MC2_OK;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const MmrsLayout L = mmrs_layout(*s);
  char* w = static_cast<char*>(ws);
  const int64_t rows = static_cast<int64_t>(s->W) * s->m;
  cudaError_t e = launch_i8_to_bf16(x1, w + L.x1_b16, static_cast<size_t>(rows) * s->k, st);
  if (e == cudaSuccess)
    e = launch_i8_to_bf16(x2, w + L.x2_b16, static_cast<size_t>(s->W) * s->k * s->n, st);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  if (e == cudaSuccess) {
    e = launch_kernel(mmrs_offsets_kernel, dim3(1), dim3(128), 0, st, 1, offsets,
                      static_cast<int>(s->W), static_cast<int>(s->m));
    if (e == cudaSuccess) note_launches(1);
  }
  // the grouped GEMM sees the ranks as groups: [W*m, k] rows against [W, k, n]
  mc2_shape_t gs;
  std::memset(&gs, 0, sizeof(gs));
  gs.T = static_cast<int32_t>(rows);
  gs.k = 1;
  gs.I = s->k;
  gs.H = s->n;
  gs.E = s->W;
  gs.W = 1;
  gs.act = MC2_I8;
  gs.out = MC2_I32;
  if (e == cudaSuccess) {
    QArgs q;
    std::memset(&q, 0, sizeof(q));
    q.s = &gs;
    q.a = w + L.x1_b16;
    q.b = w + L.x2_b16;
    q.offsets = offsets;
    q.out = w + L.acc;
    q.dev_status = dev_status;
    q.mode = MODE_FC2;
    q.raw = true;
    e = launch_gemm_q(q, st);
  }
  if (e == cudaSuccess) {
    const int64_t n = static_cast<int64_t>(s->m) * (s->n / 8);
    const int threads = 256;
    e = launch_kernel(mmrs_reduce_kernel, dim3(static_cast<unsigned>((n + threads - 1) / threads)),
                      dim3(threads), 0, st, 1, reinterpret_cast<const int32_t*>(w + L.acc), x1_scale,
                      x2_scale, static_cast<int>(s->W), static_cast<int>(s->m),
                      static_cast<int>(s->n), static_cast<__nv_bfloat16*>(out));
    if (e == cudaSuccess) note_launches(1);
  }
  return e == cudaSuccess ? MC2_OK : MC2_ERR_CUDA;
}
