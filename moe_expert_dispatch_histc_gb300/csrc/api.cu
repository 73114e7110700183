// api.cu -- the C ABI of libmc2moe: argument rules, workspace layout and the
// order of launches for each entry point.  No allocation, no synchronisation.
#include <cuda_runtime.h>

#include <cstring>
#include <initializer_list>

#include "internal.h"

namespace mc2 {

// Test and diagnostic hooks (mc2_set_*): each holds for later calls made on
// the host thread that set it, and on no other thread.  Apart from the wait
// limit, none of them changes a result bit.
static thread_local uint64_t tl_wait_limit_ns = 0;
static thread_local int tl_tile_pairing = 0;
static thread_local int tl_launch_overlap = 1;
static thread_local int tl_counts_path = 0;
static thread_local int tl_mmrs_path = 0;
static thread_local int tl_combine_path = 0;
static thread_local int tl_launches = 0;
static thread_local cudaEvent_t tl_gemm_before = nullptr;  // mc2_set_gemm_events
static thread_local cudaEvent_t tl_gemm_after = nullptr;

// Launch a call's grouped-matmul kernel, with the timing events of
// mc2_set_gemm_events recorded on its stream right before and after it.
template <class F>
static cudaError_t timed_gemm(cudaStream_t st, F&& launch) {
  if (tl_gemm_before) {
    const cudaError_t e = cudaEventRecord(tl_gemm_before, st);
    if (e != cudaSuccess) return e;
  }
  const cudaError_t e = launch();
  if (e != cudaSuccess || !tl_gemm_after) return e;
  return cudaEventRecord(tl_gemm_after, st);
}

uint64_t wait_limit_ns() { return tl_wait_limit_ns ? tl_wait_limit_ns : 2000000000ull; }  // 2 s

int tile_pairing_override() { return tl_tile_pairing; }

bool launch_overlap_enabled() { return tl_launch_overlap != 0; }

int counts_path_override() { return tl_counts_path; }

int mmrs_path_override() { return tl_mmrs_path; }

int combine_path_override() { return tl_combine_path; }

void note_launches(int n) { tl_launches += n; }

void reset_launches() { tl_launches = 0; }

WsLayout ws_layout(const mc2_shape_t& s) {
  WsLayout L;
  std::memset(&L, 0, sizeof(L));
  const CountsGeom g = counts_geom(s);
  const size_t R = static_cast<size_t>(s.T) * s.k;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kWsAlign);
    return at;
  };
  L.hist = take(static_cast<size_t>(g.EB) * g.G * 4);
  L.base = take(static_cast<size_t>(g.EB) * g.G * 4);
  L.y = take(R * s.H * 2);
  L.yscale = take(R * (s.H / 64) * 4);
  L.ctr = take(static_cast<size_t>(s.T) * ((s.H + 255) / 256) * 4);
  L.defer = take(16 + static_cast<size_t>(s.T) * ((s.H + 255) / 256) * 4);
  if (s.act == MC2_F32) {
    L.x_t32 = take(static_cast<size_t>(s.T) * s.H * 4);
    L.w1_t32 = take(static_cast<size_t>(s.E) * s.H * 2 * s.I * 4);
    L.w2_t32 = take(static_cast<size_t>(s.E) * s.I * s.H * 4);
  }
  if (s.act == MC2_I8) {
    L.x_b16 = take(static_cast<size_t>(s.T) * s.H * 2);
    L.w1_b16 = take(static_cast<size_t>(s.E) * s.H * 2 * s.I * 2);
    L.w2_b16 = take(static_cast<size_t>(s.E) * s.I * s.H * 2);
    L.h_f32 = take(R * s.I * 4);
    L.hq_b16 = take(R * s.I * 2);
  }
  L.total = off > kWsAlign ? off : kWsAlign;  // never 0: 0 means "shape rejected"
  return L;
}

}  // namespace mc2

using namespace mc2;

namespace {

bool shape_ok(const mc2_shape_t* s) {
  if (!s) return false;
  if (s->T < 0 || s->H < 64 || s->I < 64 || s->H % 64 || s->I % 64) return false;
  if (s->E < 1 || s->E > 1024 || s->k < 1 || s->k > s->E || s->W < 1) return false;
  if (s->E % s->W || s->T % s->W) return false;
  const int64_t R = static_cast<int64_t>(s->T) * s->k;
  if (R >= (int64_t(1) << 31)) return false;
  if (s->act == MC2_I8 && (s->H > 4096 || s->I > 4096)) return false;  // <= 4 exact K chunks
  const bool combo = (s->act == MC2_F32 && s->out == MC2_F32) ||
                     (s->act == MC2_BF16 && s->out == MC2_BF16) ||
                     (s->act == MC2_I8 && (s->out == MC2_BF16 || s->out == MC2_I32));
  return combo;
}

mc2_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MC2_OK : MC2_ERR_CUDA; }

mc2_status_t do_counts(const mc2_shape_t* s, const int32_t* sel, int32_t* cnt, int32_t* recv,
                       int32_t* offsets, int32_t* permute_src, int32_t* unpermute_dst, void* ws,
                       int32_t* dev_status, cudaStream_t st, bool launch = true) {
  if (!cnt || !recv || !offsets || !ws) return MC2_ERR_INVALID_ARG;
  if (s->T > 0 && (!sel || !permute_src || !unpermute_dst)) return MC2_ERR_INVALID_ARG;
  if (!aligned({sel, cnt, recv, offsets, permute_src, unpermute_dst}) || !aligned({ws}, 256))
    return MC2_ERR_INVALID_ARG;
  if (!launch) return MC2_OK;
  return cuda_status(launch_counts(*s, sel, cnt, recv, offsets, permute_src, unpermute_dst,
                                   static_cast<char*>(ws), dev_status, st));
}

mc2_status_t do_fc1_i8(const mc2_shape_t* s, const void* x, const float* x_scale,
                       const float* w1_scale, const int32_t* offsets, const int32_t* permute_src,
                       void* ws, void* h, float* h_scale, int32_t* dev_status, cudaStream_t st, bool launch = true) {
  const bool raw = s->out == MC2_I32;
  if (!offsets || !ws) return MC2_ERR_INVALID_ARG;
  // with T = 0 nothing is launched and the scales may be NULL (as the weights may)
  if (raw ? (h_scale != nullptr) : (s->T > 0 && (!w1_scale || !x_scale || !h_scale)))
    return MC2_ERR_INVALID_ARG;
  if (s->T > 0 && (!x || !permute_src || !h)) return MC2_ERR_INVALID_ARG;
  if (!aligned({x, x_scale, w1_scale, offsets, permute_src, h, h_scale}) || !aligned({ws}, 256))
    return MC2_ERR_INVALID_ARG;
  if (!launch || s->T == 0) return MC2_OK;
  const WsLayout L = ws_layout(*s);
  char* w = static_cast<char*>(ws);
  if (launch_i8_to_bf16(static_cast<const int8_t*>(x), w + L.x_b16,
                        static_cast<size_t>(s->T) * s->H, st) != cudaSuccess)
    return MC2_ERR_CUDA;
  QArgs q;
  std::memset(&q, 0, sizeof(q));
  q.s = s;
  q.a = w + L.x_b16;
  q.b = w + L.w1_b16;
  q.offsets = offsets;
  q.permute_src = permute_src;
  q.a_scale = x_scale;
  q.b_scale = w1_scale;
  q.out = raw ? h : static_cast<void*>(w + L.h_f32);
  q.dev_status = dev_status;
  q.mode = 0;
  q.raw = raw;
  cudaError_t e = timed_gemm(st, [&] { return launch_gemm_q(q, st); });
  if (e == cudaSuccess && !raw)
    e = launch_requant(reinterpret_cast<const float*>(w + L.h_f32), offsets, *s,
                       static_cast<int8_t*>(h), h_scale, st);
  return cuda_status(e);
}

mc2_status_t do_fc2_i8(const mc2_shape_t* s, const void* h, const float* h_scale,
                       const float* w2_scale, const int32_t* offsets, const int32_t* permute_src,
                       const int32_t* unpermute_dst, const float* probs, void* ws, void* out,
                       int32_t* dev_status, cudaStream_t st, bool launch = true) {
  const bool raw = s->out == MC2_I32;
  if (!offsets || !ws) return MC2_ERR_INVALID_ARG;
  if (!raw && s->T > 0 && (!w2_scale || !h_scale)) return MC2_ERR_INVALID_ARG;
  if (s->T > 0 && (!h || !permute_src || !out || (!raw && (!unpermute_dst || !probs))))
    return MC2_ERR_INVALID_ARG;
  if (!aligned({h, h_scale, w2_scale, offsets, permute_src, unpermute_dst, probs, out}) ||
      !aligned({ws}, 256))
    return MC2_ERR_INVALID_ARG;
  if (!launch || s->T == 0) return MC2_OK;
  const WsLayout L = ws_layout(*s);
  char* w = static_cast<char*>(ws);
  const size_t R = static_cast<size_t>(s->T) * s->k;
  if (launch_i8_to_bf16(static_cast<const int8_t*>(h), w + L.hq_b16, R * s->I, st) != cudaSuccess)
    return MC2_ERR_CUDA;
  QArgs q;
  std::memset(&q, 0, sizeof(q));
  q.s = s;
  q.a = w + L.hq_b16;
  q.b = w + L.w2_b16;
  q.offsets = offsets;
  q.permute_src = permute_src;
  q.a_scale = h_scale;
  q.b_scale = w2_scale;
  q.out = raw ? out : static_cast<void*>(w + L.y);
  q.yscale = reinterpret_cast<float*>(w + L.yscale);
  q.dev_status = dev_status;
  q.mode = 1;
  q.raw = raw;
  cudaError_t e = timed_gemm(st, [&] { return launch_gemm_q(q, st); });
  if (e == cudaSuccess && !raw)
    e = launch_combine(*s, w + L.y, reinterpret_cast<const float*>(w + L.yscale), probs, offsets,
                       unpermute_dst, out, MC2_BF16, st);
  return cuda_status(e);
}

mc2_status_t do_fc1(const mc2_shape_t* s, const void* x, const float* x_scale, const void* w1,
                    const float* w1_scale, const int32_t* offsets, const int32_t* permute_src,
                    void* ws, void* h, float* h_scale, int32_t* dev_status, cudaStream_t st, bool launch = true) {
  if (s->act == MC2_I8) {
    if (s->T > 0 && !w1) return MC2_ERR_INVALID_ARG;
    return do_fc1_i8(s, x, x_scale, w1_scale, offsets, permute_src, ws, h, h_scale, dev_status, st,
                     launch);
  }
  if (x_scale || w1_scale || h_scale) return MC2_ERR_INVALID_ARG;
  if (!offsets || !ws) return MC2_ERR_INVALID_ARG;
  if (s->T > 0 && (!x || !w1 || !permute_src || !h)) return MC2_ERR_INVALID_ARG;
  if (!aligned({x, w1, offsets, permute_src, h}) || !aligned({ws}, 256)) return MC2_ERR_INVALID_ARG;
  if (!launch || s->T == 0) return MC2_OK;
  const WsLayout L = ws_layout(*s);
  char* w = static_cast<char*>(ws);
  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  g.s = s;
  g.offsets = offsets;
  g.permute_src = permute_src;
  g.out = h;
  g.dev_status = dev_status;
  g.mode = MODE_FC1;
  if (s->act == MC2_F32) {
    float* xr = reinterpret_cast<float*>(w + L.x_t32);
    float* w1r = reinterpret_cast<float*>(w + L.w1_t32);
    cudaError_t e = launch_round_tf32(static_cast<const float*>(x), xr,
                                      static_cast<size_t>(s->T) * s->H, st);
    if (e == cudaSuccess)  // [E, H, 2I] -> [E, 2I, H]
      e = launch_transpose_round_tf32(static_cast<const float*>(w1), w1r, s->E, s->H, 2 * s->I, st);
    if (e != cudaSuccess) return MC2_ERR_CUDA;
    g.a = xr;
    g.b = w1r;
    g.a_elem_bytes = 4;
  } else {
    g.a = x;
    g.b = w1;
    g.a_elem_bytes = 2;
  }
  return cuda_status(timed_gemm(st, [&] { return launch_gemm(g, st); }));
}

mc2_status_t do_fc2(const mc2_shape_t* s, const void* h, const float* h_scale, const void* w2,
                    const float* w2_scale, const int32_t* offsets, const int32_t* permute_src,
                    const int32_t* unpermute_dst, const float* probs, void* ws, void* out,
                    int32_t* dev_status, cudaStream_t st, bool launch = true) {
  if (s->act == MC2_I8) {
    if (s->T > 0 && !w2) return MC2_ERR_INVALID_ARG;
    return do_fc2_i8(s, h, h_scale, w2_scale, offsets, permute_src, unpermute_dst, probs, ws, out,
                     dev_status, st, launch);
  }
  if (h_scale || w2_scale) return MC2_ERR_INVALID_ARG;
  if (!offsets || !ws) return MC2_ERR_INVALID_ARG;
  if (s->T > 0 && (!h || !w2 || !permute_src || !unpermute_dst || !probs || !out))
    return MC2_ERR_INVALID_ARG;
  if (!aligned({h, w2, offsets, permute_src, unpermute_dst, probs, out}) || !aligned({ws}, 256))
    return MC2_ERR_INVALID_ARG;
  if (!launch || s->T == 0) return MC2_OK;
  const WsLayout L = ws_layout(*s);
  char* w = static_cast<char*>(ws);
  void* y = w + L.y;
  float* yscale = reinterpret_cast<float*>(w + L.yscale);
  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  g.s = s;
  g.a = h;
  g.offsets = offsets;
  g.permute_src = permute_src;
  g.out = y;
  g.yscale = yscale;
  g.dev_status = dev_status;
  g.mode = MODE_FC2;
  if (s->act == MC2_F32) {
    float* w2r = reinterpret_cast<float*>(w + L.w2_t32);
    // [E, I, H] -> [E, H, I]
    if (launch_transpose_round_tf32(static_cast<const float*>(w2), w2r, s->E, s->I, s->H, st) !=
        cudaSuccess)
      return MC2_ERR_CUDA;
    g.b = w2r;
    g.a_elem_bytes = 4;
  } else {
    g.b = w2;
    g.a_elem_bytes = 2;
  }
  if (fused_combine_supported(*s) && combine_path_override() == 1) {
    // the fc2 kernel sums every token's rows itself as they complete
    g.mode = MODE_FC2C;
    g.probs = probs;
    g.unpermute_dst = unpermute_dst;
    g.ctr = reinterpret_cast<int32_t*>(w + L.ctr);
    g.defer_count = reinterpret_cast<int32_t*>(w + L.defer);
    g.defer_items = reinterpret_cast<int32_t*>(w + L.defer + 16);
    g.comb_out = out;
    g.out_dtype = s->out;
    return cuda_status(timed_gemm(st, [&] { return launch_gemm(g, st); }));
  }
  cudaError_t e = timed_gemm(st, [&] { return launch_gemm(g, st); });
  if (e == cudaSuccess)
    e = launch_combine(*s, y, yscale, probs, offsets, unpermute_dst, out, s->out, st);
  return cuda_status(e);
}

}  // namespace

extern "C" {

mc2_status_t mc2_check_shape(const mc2_shape_t* s) {
  return shape_ok(s) ? MC2_OK : MC2_ERR_INVALID_ARG;
}

size_t mc2_workspace_bytes(const mc2_shape_t* s) {
  if (!shape_ok(s)) return 0;
  return ws_layout(*s).total;
}

mc2_status_t mc2_moe_counts(const mc2_shape_t* s, const int32_t* sel, int32_t* cnt,
                            int32_t* recv, int32_t* offsets, int32_t* permute_src,
                            int32_t* unpermute_dst, void* ws, int32_t* dev_status,
                            void* stream) {
  tl_launches = 0;
  if (!shape_ok(s)) return MC2_ERR_INVALID_ARG;
  return do_counts(s, sel, cnt, recv, offsets, permute_src, unpermute_dst, ws, dev_status,
                   static_cast<cudaStream_t>(stream));
}

mc2_status_t mc2_alltoallv_gmm(const mc2_shape_t* s, const void* x, const float* x_scale,
                               const void* w1, const float* w1_scale, const int32_t* offsets,
                               const int32_t* permute_src, void* ws, void* h, float* h_scale,
                               int32_t* dev_status, void* stream) {
  tl_launches = 0;
  if (!shape_ok(s)) return MC2_ERR_INVALID_ARG;
  return do_fc1(s, x, x_scale, w1, w1_scale, offsets, permute_src, ws, h, h_scale, dev_status,
                static_cast<cudaStream_t>(stream));
}

mc2_status_t mc2_gmm_alltoallv(const mc2_shape_t* s, const void* h, const float* h_scale,
                               const void* w2, const float* w2_scale, const int32_t* offsets,
                               const int32_t* permute_src, const int32_t* unpermute_dst,
                               const float* probs, void* ws, void* out, int32_t* dev_status,
                               void* stream) {
  tl_launches = 0;
  if (!shape_ok(s)) return MC2_ERR_INVALID_ARG;
  return do_fc2(s, h, h_scale, w2, w2_scale, offsets, permute_src, unpermute_dst, probs, ws, out,
                dev_status, static_cast<cudaStream_t>(stream));
}

mc2_status_t mc2_moe_forward(const mc2_shape_t* s, const void* x, const float* x_scale,
                             const int32_t* sel, const float* probs, const void* w1,
                             const float* w1_scale, const void* w2, const float* w2_scale,
                             int32_t* cnt, int32_t* recv, int32_t* offsets,
                             int32_t* permute_src, int32_t* unpermute_dst, void* h,
                             float* h_scale, void* out, void* ws, int32_t* dev_status,
                             void* stream) {
  tl_launches = 0;
  if (!shape_ok(s)) return MC2_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // validate all three segments before enqueuing any of them
  for (const bool launch : {false, true}) {
    mc2_status_t r = do_counts(s, sel, cnt, recv, offsets, permute_src, unpermute_dst, ws,
                               dev_status, st, launch);
    if (r == MC2_OK)
      r = do_fc1(s, x, x_scale, w1, w1_scale, offsets, permute_src, ws, h, h_scale, dev_status,
                 st, launch);
    if (r == MC2_OK)
      r = do_fc2(s, h, h_scale, w2, w2_scale, offsets, permute_src, unpermute_dst, probs, ws,
                 out, dev_status, st, launch);
    if (r != MC2_OK) return r;
  }
  return MC2_OK;
}

mc2_status_t mc2_permute_rows(const mc2_shape_t* s, const void* x, const int32_t* permute_src,
                              void* xp, void* stream) {
  tl_launches = 0;
  if (!shape_ok(s)) return MC2_ERR_INVALID_ARG;
  if (s->T > 0 && (!x || !permute_src || !xp)) return MC2_ERR_INVALID_ARG;
  if (!aligned({x, permute_src, xp})) return MC2_ERR_INVALID_ARG;
  if (s->act != MC2_BF16) return MC2_ERR_UNSUPPORTED;
  return cuda_status(launch_permute_rows(*s, x, permute_src, xp, static_cast<cudaStream_t>(stream)));
}

mc2_status_t mc2_gmm_swiglu(const mc2_shape_t* s, const void* xp, const void* w1,
                            const int32_t* offsets, void* h, int32_t* dev_status, void* stream) {
  tl_launches = 0;
  if (!shape_ok(s)) return MC2_ERR_INVALID_ARG;
  if (!offsets) return MC2_ERR_INVALID_ARG;
  if (s->T > 0 && (!xp || !w1 || !h)) return MC2_ERR_INVALID_ARG;
  if (!aligned({xp, w1, offsets, h})) return MC2_ERR_INVALID_ARG;
  if (s->act != MC2_BF16) return MC2_ERR_UNSUPPORTED;
  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  g.s = s;
  g.a = xp;
  g.b = w1;
  g.offsets = offsets;
  g.out = h;
  g.dev_status = dev_status;
  g.mode = MODE_FC1_ROWS;
  g.a_elem_bytes = 2;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_status(timed_gemm(st, [&] { return launch_gemm(g, st); }));
}

mc2_status_t mc2_prepack_weights(const mc2_shape_t* s, const void* w1, const void* w2, void* ws,
                                 void* stream) {
  tl_launches = 0;
  if (!shape_ok(s)) return MC2_ERR_INVALID_ARG;
  if (s->act != MC2_I8) return MC2_OK;
  if (!w1 || !w2 || !ws) return MC2_ERR_INVALID_ARG;
  if (!aligned({w1, w2}) || !aligned({ws}, 256)) return MC2_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*s);
  char* w = static_cast<char*>(ws);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_status(launch_i8_to_bf16_2(static_cast<const int8_t*>(w1), w + L.w1_b16,
                                         static_cast<size_t>(s->E) * s->H * 2 * s->I,
                                         static_cast<const int8_t*>(w2), w + L.w2_b16,
                                         static_cast<size_t>(s->E) * s->I * s->H, st));
}

mc2_status_t mc2_selftest_wait(uint64_t limit_ns, int32_t* dev_status, void* stream) {
  tl_launches = 0;
  if (!dev_status) return MC2_ERR_INVALID_ARG;
  return cuda_status(launch_selftest_wait(limit_ns, dev_status, static_cast<cudaStream_t>(stream)));
}

void mc2_set_wait_limit_ns(uint64_t limit_ns) { tl_wait_limit_ns = limit_ns; }

void mc2_set_tile_pairing(int32_t mode) { tl_tile_pairing = mode >= 1 && mode <= 2 ? mode : 0; }

void mc2_set_launch_overlap(int32_t enabled) { tl_launch_overlap = enabled ? 1 : 0; }

void mc2_set_counts_path(int32_t mode) { tl_counts_path = mode == 1 || mode == 2 ? mode : 0; }

void mc2_set_mmrs_path(int32_t mode) { tl_mmrs_path = mode == 1 ? 1 : 0; }

void mc2_set_combine_path(int32_t mode) { tl_combine_path = mode == 1 ? 1 : 0; }

void mc2_set_gemm_events(void* before, void* after) {
  tl_gemm_before = static_cast<cudaEvent_t>(before);
  tl_gemm_after = static_cast<cudaEvent_t>(after);
}

int32_t mc2_last_launch_count(void) { return tl_launches; }

const char* mc2_status_str(mc2_status_t st) {
  switch (st) {
    case MC2_OK: return "ok";
    case MC2_ERR_INVALID_ARG: return "invalid argument";
    case MC2_ERR_UNSUPPORTED: return "unsupported";
    case MC2_ERR_CUDA: return "CUDA error";
    case MC2_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MC2_ERR_BAD_EXPERT_ID: return "expert id outside [0, E)";
  }
  return "unknown status";
}

}  // extern "C"
