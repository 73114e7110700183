// gmm_common.cuh -- tile constants, parameter block and device/host helpers
// shared by the grouped-GEMM kernels (bf16/tf32 in gmm.cu, int8 in gmm_q.cu).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace mc2 {


constexpr int BM = 128;            // rows per tile (UMMA M)
constexpr int BN = 256;            // accumulator columns per tile (UMMA N)
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * 128;  // 128 rows x 128 bytes of K
constexpr int B_STAGE = 32768;     // (128/es) K rows x 256 columns x es bytes
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int TMEM_COLS = 512;
constexpr int OUT_STAGE = 4096;    // epilogue staging per warp: 32 rows x 128 bytes

struct GemmParams {
  const void* a_ptr;            // fc1: x (rows gathered by the gather warps)
  const int32_t* offsets;
  const int32_t* permute_src;
  void* out;                    // fc1: h [R, I]; fc2: y [R, H] fp16 (scaled)
  float* yscale;                // fc2: decode factor per (row, 64 columns) [R, H/64]
  int32_t* dev_status;
  // fc2 with the combine fused (MODE_FC2C)
  const float* probs;           // routing weights [T, k]
  const int32_t* unpermute_dst; // [T*k]
  int32_t* ctr;                 // arrivals per (token, BN-column tile) [T, n_tiles]
  int32_t* defer_items;         // (token, column tile) sums left to combine_deferred_kernel
  int32_t* defer_count;         // number of deferred items
  void* comb_out;               // the block output [T, H], bf16 or fp32
  int out_f32;
  int E, k, K, n_tiles, out_cols, I;
  uint64_t wait_limit_ns;
};

template <int ES>
struct ElemTraits;
template <>
struct ElemTraits<2> {  // bf16, kind::f16; weights used as stored ([K, N], N contiguous)
  static constexpr int BK = 64;
  static constexpr int KIND = 0;
  static constexpr uint32_t FMT = 1;
  static constexpr bool B_KMAJOR = false;
};
template <>
struct ElemTraits<4> {  // fp32 storage, kind::tf32; weights pre-transposed to [N, K]
  static constexpr int BK = 32;
  static constexpr int KIND = 1;
  static constexpr uint32_t FMT = 2;
  static constexpr bool B_KMAJOR = true;
};

__device__ __forceinline__ void decode_tile(int tile, const int32_t* prefix, int E, int n_tiles,
                                            const int32_t* offsets, int& e, int& n, int& row0,
                                            int& rows) {
  int lo = 0, hi = E;  // prefix[lo] <= tile < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  e = lo;
  const int local = tile - prefix[e];
  const int m_tiles = (prefix[e + 1] - prefix[e]) / n_tiles;
  n = local / m_tiles;
  const int m = local - n * m_tiles;
  const int off = __ldg(offsets + e);
  row0 = off + m * BM;
  const int end = __ldg(offsets + e + 1);
  rows = min(BM, end - row0);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 64 fp32 values of one row (a: columns 0-31, b: 32-63) -> 64 fp16 values
// scaled by a power of two 2^se that puts max|y| in [2^14, 2^15) (fp16 has
// 11 significant bits, so each value keeps a relative error <= 2^-11).
// Returns the exact decode factor 2^-se.
__device__ __forceinline__ float pack_y16(const uint32_t (&a)[32], const uint32_t (&b)[32],
                                          uint32_t (&pk)[32]) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    m = fmaxf(m, fmaxf(fabsf(__uint_as_float(a[i])), fabsf(__uint_as_float(b[i]))));
  const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xffu) - 126;  // m = f * 2^e
  const int se = max(-126, min(126, 15 - e));
  const float scale = __uint_as_float(static_cast<uint32_t>(127 + se) << 23);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    pk[i] = pack_half2(__uint_as_float(a[2 * i]) * scale, __uint_as_float(a[2 * i + 1]) * scale);
    pk[16 + i] =
        pack_half2(__uint_as_float(b[2 * i]) * scale, __uint_as_float(b[2 * i + 1]) * scale);
  }
  return __uint_as_float(static_cast<uint32_t>(127 - se) << 23);
}

__device__ __forceinline__ float round_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// silu(g) = g / (1 + e^-g) with the fast exponential and division
// (relative error of a few fp32 ulp, far below the bf16 rounding of h).
// For g << 0, e^-g overflows to +inf and the quotient is -0.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// ----------------------------------------------------------------------------
// host: tensor maps (the driver entry point is looked up at run time)
// ----------------------------------------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

inline bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, int es, const void* base,
                      uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * es};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, int es, const void* base,
                      uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major bf16 weights [E, K, N] seen as blocks of 64 columns (128 bytes):
// dims (64, K, N/64 [, halves], E).  With halves = 2 the N columns are two
// halves of N/2 (fc1's gate and up projections) and the map's block index
// runs within one half, so one box can take the same 128 output columns of
// both halves.  A box of (64, bk, nblk [, nhalf], 1) lands in shared memory as
// [half][block][k row][128 B], each 64 x 128 B block 128-byte swizzled: the
// MN-major UMMA operand layout, in one TMA instruction instead of one per
// block.  Requires N % 64 == 0 (N/2 % 64 == 0 with halves).
inline bool encode_b_blocked(CUtensorMap* m, const void* base, uint64_t K, uint64_t N, uint64_t E,
                             int halves, uint32_t bk, uint32_t nblk, uint32_t nhalf) {
  auto enc = get_encode();
  if (!enc) return false;
  const uint64_t row = N * 2;  // bytes per k row
  if (halves == 2) {
    cuuint64_t dims[5] = {64, K, N / 2 / 64, 2, E};
    cuuint64_t strides[4] = {row, 128, N, K * row};  // half stride: N/2 columns = N bytes
    cuuint32_t box[5] = {64, bk, nblk, nhalf, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  cuuint64_t dims[4] = {64, K, N / 64, E};
  cuuint64_t strides[3] = {row, 128, K * row};
  cuuint32_t box[4] = {64, bk, nblk, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mc2
