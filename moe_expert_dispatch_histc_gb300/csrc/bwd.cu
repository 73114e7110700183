// bwd.cu -- backward of the MoE expert block (bf16): the chain rule of the
// forward flow of "NPU Training Operators - MC2", section "Execution path",
// steps 10 back to 6, for L = sum(out * dout):
//
//   D[p]      = dout[t(p)]                       gathered output gradient rows
//   dhu[p]    = D[p] @ w2[e]^T                   (fc2 kernel on w2 transposed)
//   dprobs    = h[p] . dhu[p]                    (= Y[p] . dout[t])
//   dh[p]     = probs[t, j] * dhu[p]
//   dG        = [dh * up * silu'(gate), dh * silu(gate)]     G = x[t] @ w1[e]
//   dXp[p]    = dG[p] @ w1[e]^T                  (fc2 kernel on w1 transposed)
//   dx[t]     = sum over t's valid slots of dXp  (the combine with unit weights)
//   dw2[e]    = (probs * h)_e^T @ D_e ;  dw1[e] = Xp_e^T @ dG_e    (wgrad.cu)
//
// G is recomputed (the fc1 kernel in its pre-activation mode) and h from G,
// so the backward needs only the forward's inputs and the counts outputs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <initializer_list>

#include "gmm_common.cuh"

namespace mc2 {
namespace {

struct BwdLayout {
  size_t xp, g, d, dhu, dhs, dg, hp, dxp, dxs, ones, total;
};

BwdLayout bwd_layout(const mc2_shape_t& s) {
  BwdLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kWsAlign);
    return at;
  };
  const size_t R = static_cast<size_t>(s.T) * s.k, H = s.H, I = s.I;
  L.xp = take(R * H * 2);       // bf16 permuted x rows
  L.g = take(R * 2 * I * 2);    // bf16 pre-activation gate | up
  L.d = take(R * H * 2);        // bf16 gathered dout rows
  L.dhu = take(R * I * 2);      // fp16 rows of D @ w2^T (scaled)
  L.dhs = take(R * (I / 64) * 4);
  L.dg = take(R * 2 * I * 2);   // bf16 dG
  L.hp = take(R * I * 2);       // bf16 probs * h
  L.dxp = take(R * H * 2);      // fp16 rows of dG @ w1^T (scaled)
  L.dxs = take(R * (H / 64) * 4);
  L.ones = take(static_cast<size_t>(s.T) * s.k * 4);
  L.total = off > kWsAlign ? off : kWsAlign;
  return L;
}

// dst[b, c, r] = src[b, r, c] for bf16 [batch, rows, cols]
__global__ void transpose_bf16_kernel(const __nv_bfloat16* __restrict__ src,
                                      __nv_bfloat16* __restrict__ dst, int rows, int cols) {
  __shared__ __nv_bfloat16 tile[32][34];
  griddep_wait();
  griddep_launch_dependents();
  const int64_t b = blockIdx.z;
  const __nv_bfloat16* s = src + b * rows * static_cast<int64_t>(cols);
  __nv_bfloat16* d = dst + b * rows * static_cast<int64_t>(cols);
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = s[static_cast<int64_t>(r) * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) d[static_cast<int64_t>(c) * rows + r] = tile[threadIdx.x][i];
  }
}

__global__ void fill_f32_kernel(float* __restrict__ p, int64_t n, float v) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) p[i] = v;
}

__device__ __forceinline__ float sigmoid_f(float a) { return 1.0f / (1.0f + expf(-a)); }

// Training forward: h[p] = bf16(silu(gate) * up) from the kept pre-activation
// rows G [R, 2I] (bf16), rows p < offsets[E]; 8 columns per thread.
__global__ void swiglu_fwd_kernel(const __nv_bfloat16* __restrict__ G,
                                  const int32_t* __restrict__ offsets, int E, int I,
                                  __nv_bfloat16* __restrict__ h) {
  griddep_wait();
  griddep_launch_dependents();
  const int I8 = I / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t p = idx / I8;
  if (p >= __ldg(offsets + E)) return;
  const int c = static_cast<int>(idx - p * I8) * 8;
  const uint4 ga = __ldg(reinterpret_cast<const uint4*>(G + p * 2 * I + c));
  const uint4 ua = __ldg(reinterpret_cast<const uint4*>(G + p * 2 * I + I + c));
  const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&ga);
  const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&ua);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 gv = __bfloat1622float2(g2[i]);
    const float2 uv = __bfloat1622float2(u2[i]);
    o[i] = pack_bf16x2(silu_f(gv.x) * uv.x, silu_f(gv.y) * uv.y);
  }
  *reinterpret_cast<uint4*>(h + p * I + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

// One warp per permuted row p.  Valid rows: dG, probs * h and dprobs of the
// row's (token, slot).  Rows of invalid ids: dprobs of their slot = 0, and
// zero dG and probs * h rows (the weight-gradient GEMM may read them as the
// rows after the last expert; zero keeps whatever was in the workspace out).
__global__ void swiglu_bwd_kernel(const __nv_bfloat16* __restrict__ G,
                                  const __half* __restrict__ dhu, const float* __restrict__ dhs,
                                  const float* __restrict__ probs,
                                  const int32_t* __restrict__ offsets,
                                  const int32_t* __restrict__ permute_src, int64_t R, int E, int I,
                                  __nv_bfloat16* __restrict__ dG, __nv_bfloat16* __restrict__ hp,
                                  float* __restrict__ dprobs) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t p = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (p >= R) return;
  const int32_t flat = __ldg(permute_src + p);
  if (p >= __ldg(offsets + E)) {
    if (lane == 0) dprobs[flat] = 0.f;
    for (int c = lane * 8; c < I; c += 256) {
      *reinterpret_cast<uint4*>(dG + p * 2 * I + c) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(dG + p * 2 * I + I + c) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(hp + p * I + c) = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const float pj = __ldg(probs + flat);
  const __nv_bfloat16* g = G + p * 2 * I;
  float dot = 0.f;
  for (int c = lane * 8; c < I; c += 256) {
    const uint4 ga = __ldg(reinterpret_cast<const uint4*>(g + c));
    const uint4 ua = __ldg(reinterpret_cast<const uint4*>(g + I + c));
    const uint4 da = __ldg(reinterpret_cast<const uint4*>(dhu + p * I + c));
    const float f = __ldg(dhs + p * (I / 64) + c / 64);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&ga);
    const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&ua);
    const __half2* d2 = reinterpret_cast<const __half2*>(&da);
    uint32_t og[4], ou[4], oh[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 gv = __bfloat1622float2(g2[i]);
      const float2 uv = __bfloat1622float2(u2[i]);
      const float2 dv = __half22float2(d2[i]);
      float rg[2], ru[2], rh[2];
      const float gg[2] = {gv.x, gv.y}, uu[2] = {uv.x, uv.y}, dd[2] = {dv.x * f, dv.y * f};
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float sg = sigmoid_f(gg[q]);
        const float si = gg[q] * sg;
        // h as the forward materialises it: bf16(silu(gate) * up)
        const float h = __bfloat162float(__float2bfloat16_rn(si * uu[q]));
        dot += h * dd[q];
        const float dh = pj * dd[q];
        rg[q] = dh * uu[q] * (sg * (1.0f + gg[q] * (1.0f - sg)));
        ru[q] = dh * si;
        rh[q] = pj * h;
      }
      og[i] = pack_bf16x2(rg[0], rg[1]);
      ou[i] = pack_bf16x2(ru[0], ru[1]);
      oh[i] = pack_bf16x2(rh[0], rh[1]);
    }
    *reinterpret_cast<uint4*>(dG + p * 2 * I + c) = make_uint4(og[0], og[1], og[2], og[3]);
    *reinterpret_cast<uint4*>(dG + p * 2 * I + I + c) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
    *reinterpret_cast<uint4*>(hp + p * I + c) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  if (lane == 0) dprobs[flat] = dot;
}

bool al(std::initializer_list<const void*> ps, uintptr_t a = 16) {
  for (const void* p : ps)
    if (reinterpret_cast<uintptr_t>(p) & (a - 1)) return false;
  return true;
}

bool bwd_shape_ok(const mc2_shape_t* s) {
  return mc2_check_shape(s) == MC2_OK && s->act == MC2_BF16 && s->out == MC2_BF16;
}

}  // namespace
}  // namespace mc2

using namespace mc2;

extern "C" size_t mc2_backward_workspace_bytes(const mc2_shape_t* s) {
  if (!bwd_shape_ok(s)) return 0;
  return bwd_layout(*s).total;
}

extern "C" mc2_status_t mc2_transpose_weights(const mc2_shape_t* s, const void* w1,
                                              const void* w2, void* w1t, void* w2t,
                                              void* stream) {
  reset_launches();
  if (mc2_check_shape(s) != MC2_OK) return MC2_ERR_INVALID_ARG;
  if (s->act != MC2_BF16) return MC2_ERR_UNSUPPORTED;
  if (!w1 || !w2 || !w1t || !w2t || !al({w1, w2, w1t, w2t})) return MC2_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // w1 [E, H, 2I] -> w1t [E, 2I, H];  w2 [E, I, H] -> w2t [E, H, I]
  const dim3 blk(32, 8);
  cudaError_t e = launch_kernel(transpose_bf16_kernel, dim3((2 * s->I + 31) / 32, (s->H + 31) / 32,
                                                            s->E),
                                blk, 0, st, 1, static_cast<const __nv_bfloat16*>(w1),
                                static_cast<__nv_bfloat16*>(w1t), static_cast<int>(s->H),
                                static_cast<int>(2 * s->I));
  if (e == cudaSuccess)
    e = launch_kernel(transpose_bf16_kernel, dim3((s->H + 31) / 32, (s->I + 31) / 32, s->E), blk, 0,
                      st, 1, static_cast<const __nv_bfloat16*>(w2), static_cast<__nv_bfloat16*>(w2t),
                      static_cast<int>(s->I), static_cast<int>(s->H));
  if (e == cudaSuccess) note_launches(2);
  return e == cudaSuccess ? MC2_OK : MC2_ERR_CUDA;
}

extern "C" mc2_status_t mc2_alltoallv_gmm_keep(const mc2_shape_t* s, const void* x,
                                               const void* w1, const int32_t* offsets,
                                               const int32_t* permute_src, void* h, void* g,
                                               int32_t* dev_status, void* stream) {
  reset_launches();
  if (mc2_check_shape(s) != MC2_OK) return MC2_ERR_INVALID_ARG;
  if (!bwd_shape_ok(s)) return MC2_ERR_UNSUPPORTED;
  if (!offsets) return MC2_ERR_INVALID_ARG;
  if (s->T > 0 && (!x || !w1 || !permute_src || !h || !g)) return MC2_ERR_INVALID_ARG;
  if (!al({x, w1, offsets, permute_src, h, g})) return MC2_ERR_INVALID_ARG;
  const int64_t R = static_cast<int64_t>(s->T) * s->k;
  if (R == 0) return MC2_OK;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.s = s;
  a.a = x;
  a.b = w1;
  a.offsets = offsets;
  a.permute_src = permute_src;
  a.out = g;
  a.dev_status = dev_status;
  a.mode = MODE_FC1_PRE;
  a.a_elem_bytes = 2;
  cudaError_t e = launch_gemm(a, st);
  if (e == cudaSuccess) {
    const int64_t n = R * (s->I / 8);
    e = launch_kernel(swiglu_fwd_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0,
                      st, 1, static_cast<const __nv_bfloat16*>(g), offsets, static_cast<int>(s->E),
                      static_cast<int>(s->I), static_cast<__nv_bfloat16*>(h));
    if (e == cudaSuccess) note_launches(1);
  }
  return e == cudaSuccess ? MC2_OK : MC2_ERR_CUDA;
}

extern "C" mc2_status_t mc2_moe_backward(const mc2_shape_t* s, const void* x, const float* probs,
                                         const void* w1, const void* g_kept, const void* w1t,
                                         const void* w2t,
                                         const void* dout, const int32_t* offsets,
                                         const int32_t* permute_src,
                                         const int32_t* unpermute_dst, void* dx, float* dw1,
                                         float* dw2, float* dprobs, void* ws,
                                         int32_t* dev_status, void* stream) {
  reset_launches();
  if (mc2_check_shape(s) != MC2_OK) return MC2_ERR_INVALID_ARG;
  if (!bwd_shape_ok(s)) return MC2_ERR_UNSUPPORTED;
  if (!offsets || !ws || !w1 || !w1t || !w2t || !dw1 || !dw2) return MC2_ERR_INVALID_ARG;
  if (s->T > 0 && (!x || !probs || !dout || !permute_src || !unpermute_dst || !dx || !dprobs))
    return MC2_ERR_INVALID_ARG;
  if (!al({x, probs, w1, g_kept, w1t, w2t, dout, offsets, permute_src, unpermute_dst, dx, dw1,
           dw2, dprobs}) ||
      !al({ws}, 256))
    return MC2_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t R = static_cast<int64_t>(s->T) * s->k;
  const BwdLayout L = bwd_layout(*s);
  char* w = static_cast<char*>(ws);
  auto* xp = w + L.xp;
  const void* G = g_kept ? g_kept : static_cast<const void*>(w + L.g);
  auto* D = w + L.d;
  auto* dhu = w + L.dhu;
  auto* dhs = reinterpret_cast<float*>(w + L.dhs);
  auto* dG = w + L.dg;
  auto* hp = w + L.hp;
  auto* dxp = w + L.dxp;
  auto* dxs = reinterpret_cast<float*>(w + L.dxs);
  auto* ones = reinterpret_cast<float*>(w + L.ones);
  cudaError_t e = cudaSuccess;
  if (R > 0) {
    // G (pre-activation gate | up): kept by the training forward, else recomputed
    // with the fc1 kernel; then the permuted rows of x and dout
    if (!g_kept) {
      GemmArgs g;
      std::memset(&g, 0, sizeof(g));
      g.s = s;
      g.a = x;
      g.b = w1;
      g.offsets = offsets;
      g.permute_src = permute_src;
      g.out = w + L.g;
      g.dev_status = dev_status;
      g.mode = MODE_FC1_PRE;
      g.a_elem_bytes = 2;
      e = launch_gemm(g, st);
    }
    if (e == cudaSuccess) e = launch_permute_rows(*s, x, permute_src, xp, st);
    if (e == cudaSuccess) e = launch_permute_rows(*s, dout, permute_src, D, st);
    // dhu = D @ w2^T: the fc2 kernel with K = H, N = I on w2t [E, H, I]
    mc2_shape_t s2 = *s;
    s2.I = s->H;
    s2.H = s->I;
    if (e == cudaSuccess) {
      GemmArgs d2;
      std::memset(&d2, 0, sizeof(d2));
      d2.s = &s2;
      d2.a = D;
      d2.b = w2t;
      d2.offsets = offsets;
      d2.permute_src = permute_src;
      d2.out = dhu;
      d2.yscale = dhs;
      d2.dev_status = dev_status;
      d2.mode = MODE_FC2;
      d2.a_elem_bytes = 2;
      e = launch_gemm(d2, st);
    }
    if (e == cudaSuccess) {
      const int warps = 8;
      e = launch_kernel(swiglu_bwd_kernel, dim3(static_cast<unsigned>((R + warps - 1) / warps)),
                        dim3(warps * 32), 0, st, 1, static_cast<const __nv_bfloat16*>(
                            static_cast<const void*>(G)),
                        static_cast<const __half*>(static_cast<const void*>(dhu)), dhs, probs,
                        offsets, permute_src, R, static_cast<int>(s->E), static_cast<int>(s->I),
                        static_cast<__nv_bfloat16*>(static_cast<void*>(dG)),
                        static_cast<__nv_bfloat16*>(static_cast<void*>(hp)), dprobs);
      if (e == cudaSuccess) note_launches(1);
    }
    // dXp = dG @ w1^T: the fc2 kernel with K = 2I, N = H on w1t [E, 2I, H]
    mc2_shape_t s1 = *s;
    s1.I = 2 * s->I;
    s1.H = s->H;
    if (e == cudaSuccess) {
      GemmArgs d1;
      std::memset(&d1, 0, sizeof(d1));
      d1.s = &s1;
      d1.a = dG;
      d1.b = w1t;
      d1.offsets = offsets;
      d1.permute_src = permute_src;
      d1.out = dxp;
      d1.yscale = dxs;
      d1.dev_status = dev_status;
      d1.mode = MODE_FC2;
      d1.a_elem_bytes = 2;
      e = launch_gemm(d1, st);
    }
    // dx = the combine with unit weights
    if (e == cudaSuccess) {
      e = launch_kernel(fill_f32_kernel, dim3(static_cast<unsigned>((R + 255) / 256)), dim3(256), 0,
                        st, 1, ones, R, 1.0f);
      if (e == cudaSuccess) note_launches(1);
    }
    if (e == cudaSuccess)
      e = launch_combine(*s, dxp, dxs, ones, offsets, unpermute_dst, dx, MC2_BF16, st);
  }
  // weight gradients (written for every expert, zero where an expert has no rows)
  if (e == cudaSuccess)
    e = launch_wgrad(hp, D, offsets, R, s->E, s->I, s->H, dw2, dev_status, st);
  if (e == cudaSuccess)
    e = launch_wgrad(xp, dG, offsets, R, s->E, s->H, 2 * s->I, dw1, dev_status, st);
  return e == cudaSuccess ? MC2_OK : MC2_ERR_CUDA;
}
