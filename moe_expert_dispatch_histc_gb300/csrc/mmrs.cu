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
// rank index and a row split.  The int8 values run exactly on the bf16 tensor
// cores (int8 -> bf16 copies first; K summed in exact fp32 chunks of 1024, as
// in gmm_q.cu).  Two forms give the same bits:
//   fused (default): mmrs_fused_kernel, one CTA-pair kernel per call that
//     keeps every output tile's rank sum on chip (below);
//   two passes: the exact int8 grouped GEMM of the MoE block (gmm_q.cu, raw
//     int32 accumulators, one group per rank: rows r*m .. r*m+m-1 of the
//     stacked x1 against x2_r) writes every rank's partial product to the
//     workspace, then mmrs_reduce_kernel sums the dequantised partials.
// Both fold rank r in as fma(x1_scale * x2_scale, float(acc), sum) in fp32,
// r ascending, and round once to bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "gmm_common.cuh"

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

// out[i, c..c+7] = bf16( sum_r (xs[r, i] * ws[r, c]) * float(acc[r*m + i, c]) ), r ascending,
// each rank folded in with one fma
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
    s[0] = __fmaf_rn(xr * w0.x, static_cast<float>(a0.x), s[0]);
    s[1] = __fmaf_rn(xr * w0.y, static_cast<float>(a0.y), s[1]);
    s[2] = __fmaf_rn(xr * w0.z, static_cast<float>(a0.z), s[2]);
    s[3] = __fmaf_rn(xr * w0.w, static_cast<float>(a0.w), s[3]);
    s[4] = __fmaf_rn(xr * w1.x, static_cast<float>(a1.x), s[4]);
    s[5] = __fmaf_rn(xr * w1.y, static_cast<float>(a1.y), s[5]);
    s[6] = __fmaf_rn(xr * w1.z, static_cast<float>(a1.z), s[6]);
    s[7] = __fmaf_rn(xr * w1.w, static_cast<float>(a1.w), s[7]);
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

// ----------------------------------------------------------------------------
// Fused form: one CTA-pair kernel (tcgen05 cta_group::2, UMMA M = 256, N = NB).
// A cluster owns an output tile of 256 rows x NB columns (each CTA 128 rows).
// For every rank r in ascending order it accumulates x1_r @ x2_r into TMEM
// (K in exact chunks of 1024, one accumulator region each), and the epilogue
// warps fold (x1_scale_r * x2_scale_r) * acc_r into an fp32 running sum held
// in registers: one row and 128 columns per thread (NB / 32 epilogue warps).
// Two TMEM accumulator sets, when they fit, let rank r+1's MMAs run while
// rank r is folded in.  After the last rank the sum is rounded to bf16 and
// stored with TMA: the int32 partials never leave the SM, and the arithmetic
// is that of the two-pass form, so both give the same bits.  Both CTAs'
// operand loads of a stage complete on the even CTA's barrier (the odd CTA
// uses the pair form of the TMA copy), so the even CTA's MMA thread starts a
// stage as soon as both halves have landed, with no relay through the odd CTA.
//   NB = 256 (K <= 2048): 32 KB per CTA per 64-deep stage for 128 x 256 x 64
//     MMAs, six stages, eight epilogue warps;
//   NB = 128 (any K up to 4096): 24 KB per stage for 128 x 128 x 64, eight
//     stages, four epilogue warps.
// ----------------------------------------------------------------------------
constexpr int F_A_STAGE = 128 * 128;         // 128 rows x 64 K values x 2 B
constexpr int F_OUT_STAGE = 32 * 128;        // per epilogue warp: 32 rows x 64 bf16
constexpr int F_CHUNK_KB = 16;               // k-blocks of 64 per exact fp32 chunk (K 1024)
constexpr uint32_t F_TMEM_COLS = 512;

template <int NB>
struct FCfg {
  static constexpr int kEpiWarps = NB / 32;             // 128 columns per epilogue thread
  static constexpr int kThreads = (2 + kEpiWarps) * 32;  // producer, MMA, epilogue
  static constexpr int kStages = NB == 256 ? 6 : 8;
  static constexpr int kBStage = 64 * (NB / 2) * 2;      // 64 K rows x this CTA's NB/2 columns
  static constexpr int kStageBytes = F_A_STAGE + kBStage;
  static constexpr int kGW = NB == 256 ? 8 : 32;        // epilogue column group (registers)
  static constexpr size_t kSmem =
      1024 + static_cast<size_t>(kStages) * kStageBytes + kEpiWarps * F_OUT_STAGE + 256;
};

struct FParams {
  const float* xs;       // x1_scale [W, m]
  const float* ws;       // x2_scale [W, n]
  int32_t* dev_status;
  int W, m, n, K, n_tiles, m_tiles, total, nchunk;
  uint64_t wait_limit_ns;
};

// Output tile order: groups of MMRS_GROUP_M row blocks, and within a group
// the row block varies fastest.  The clusters running at the same time then
// share the x1 row blocks and x2 column blocks they stream (for every rank)
// and consecutive waves reuse row blocks from L2.  Measured on GB300 at W8
// m4096 k1024 n4096 (16 row blocks): groups of 2 / 4 / 8 / 16 row blocks
// 0.255 / 0.252 / 0.248 / 0.246 ms per call, plain row-major order 0.255;
// the kernel's DRAM reads 280 MB with 8 against 328 MB with 16.
constexpr int MMRS_GROUP_M = 8;

__device__ __forceinline__ void mmrs_tile(int tile, int m_tiles, int n_tiles, int& mt, int& nt) {
  const int per_group = MMRS_GROUP_M * n_tiles;
  const int g = tile / per_group;
  const int first = g * MMRS_GROUP_M;
  const int gm = min(MMRS_GROUP_M, m_tiles - first);
  const int local = tile - g * per_group;
  mt = first + local % gm;
  nt = local / gm;
}

template <int GW>
__device__ __forceinline__ void tmem_ld_group(uint32_t taddr, uint32_t (&v)[GW]) {
  if constexpr (GW == 32) tmem_ld32(taddr, v);
  else if constexpr (GW == 16) tmem_ld16(taddr, v);
  else tmem_ld8(taddr, v);
}

template <int NB>
__global__ void __launch_bounds__(FCfg<NB>::kThreads, 1)
    mmrs_fused_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmOut, const FParams p) {
  using C = FCfg<NB>;
  constexpr int BK = 64;
  constexpr int STAGES = C::kStages;
  constexpr int B_STAGE = C::kBStage;
  constexpr int GW = C::kGW;
  constexpr int KK_B = 16 * 128;             // B bytes per UMMA K step (16 K rows)
  constexpr uint32_t IDESC = instr_desc(1, false, true, 256, NB);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * F_A_STAGE;
  uint8_t* sOut = sB + STAGES * B_STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + C::kEpiWarps * F_OUT_STAGE);  // even CTA
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_sh = reinterpret_cast<volatile int*>(tmem_base_sh + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int nchunk = p.nchunk;
  const uint32_t acc_cols = static_cast<uint32_t>(nchunk * NB);
  const int bufs = 2 * acc_cols <= F_TMEM_COLS ? 2 : 1;  // accumulator sets that fit

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * C::kEpiWarps);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(mma_done, 1);
    *abort_sh = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_base_sh, F_TMEM_COLS);
    tmem_relinquish_pair();
  }
  griddep_wait();
  griddep_launch_dependents();
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_sh;
  // the pair's MMAs write one TMEM address in both CTAs
  const uint32_t peer_base = ld_shared_cluster_u32(map_to_rank(tmem_base_sh, rank ^ 1u));
  int total = p.total;
  if (peer_base != tmem_base) {
    if (threadIdx.x == 0 && p.dev_status) atomicOr(p.dev_status, 0x4);
    total = 0;
  }
  WaitCtl ctl{abort_sh, p.wait_limit_ns, p.dev_status};
  const int kblocks = p.K / BK;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Both CTAs' loads of a stage complete on the even CTA's full[s] (the even
    // producer expects the bytes of both halves); the odd CTA loads with the
    // pair form of the copy, straight onto that barrier.
    const uint32_t leader_full = map_to_rank(full, 0);
    int s = 0;
    uint32_t ph = 0;
    int n_arm = 0;
    bool ok = true;
    for (int tile = cluster; tile < total && ok; tile += nclusters) {
      int mt, nt;
      mmrs_tile(tile, p.m_tiles, p.n_tiles, mt, nt);
      const int row0 = mt * 256 + static_cast<int>(rank) * 128;     // row within a rank's x1
      const int col0 = nt * NB + static_cast<int>(rank) * (NB / 2);  // this CTA's half of B
      for (int r = 0; r < p.W && ok; ++r) {
        for (int kb = 0; kb < kblocks; ++kb) {
          if (lane == 0) ok = mbar_wait_cluster(&empty[s], ph ^ 1, ctl);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (lane == 0) {
            uint8_t* a_dst = sA + s * F_A_STAGE;
            uint8_t* b_dst = sB + s * B_STAGE;
            if (leader) {
              mbar_arrive_expect_tx(&full[s], 2 * C::kStageBytes);
              tma_load_2d(a_dst, &tmA, &full[s], kb * BK, r * p.m + row0);
#pragma unroll
              for (int j = 0; j < NB / 128; ++j)   // 64-column blocks, 8 KB apart
                tma_load_3d(b_dst + j * 8192, &tmB, &full[s], col0 + 64 * j, kb * BK, r);
            } else {
              const uint32_t bar = leader_full + s * 8;
              tma_load_2d_pair(a_dst, &tmA, bar, kb * BK, r * p.m + row0);
#pragma unroll
              for (int j = 0; j < NB / 128; ++j)
                tma_load_3d_pair(b_dst + j * 8192, &tmB, bar, col0 + 64 * j, kb * BK, r);
            }
          }
          __syncwarp();
          ++n_arm;
          if (++s == STAGES) { s = 0; ph ^= 1; }
        }
      }
    }
    if (lane == 0) {  // every armed stage has landed and every commit to it has arrived
      volatile int never = 0;
      WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
      for (int st = 0; st < STAGES && st < n_arm; ++st) {
        const int last = st + STAGES * ((n_arm - 1 - st) / STAGES);
        if (leader) mbar_wait_cluster(&full[st], (last / STAGES) & 1, drain);
        mbar_wait_cluster(&empty[st], (last / STAGES) & 1, drain);
      }
    }
  } else if (warp == 1) {
    if (leader) {
      // ---------------------------------------------------------- MMA issuer
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int tile = cluster; tile < total && ok; tile += nclusters) {
        for (int r = 0; r < p.W && ok; ++r) {
          if (lane == 0) ok = mbar_wait_cluster(&tempty[acc], aph ^ 1, ctl);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d0 = tmem_base + acc * acc_cols;
          for (int kb = 0; kb < kblocks; ++kb) {
            if (lane == 0) ok = mbar_wait_cluster(&full[s], ph, ctl);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
              const uint32_t a_base = smem_u32(sA + s * F_A_STAGE);
              const uint32_t b_base = smem_u32(sB + s * B_STAGE);
              const uint32_t d = d0 + static_cast<uint32_t>((kb / F_CHUNK_KB) * NB);
              const bool first = (kb % F_CHUNK_KB) == 0;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
                const uint64_t bdesc = smem_desc_sw128(b_base + kk * KK_B, 8192, 1024);
                umma_pair<0>(d, adesc, bdesc, IDESC, (first && kk == 0) ? 0u : 1u);
              }
              umma_commit_pair(&empty[s], 0x3);
            }
            __syncwarp();
            if (++s == STAGES) { s = 0; ph ^= 1; }
          }
          if (!ok) break;
          if (lane == 0) umma_commit_pair(&tfull[acc], 0x3);
          __syncwarp();
          if (bufs == 2) acc ^= 1;
          if (acc == 0) aph ^= 1;
        }
      }
      if (lane == 0) {
        umma_commit_pair(mma_done, 0x1);
        volatile int never = 0;
        WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
        mbar_wait_cluster(mma_done, 0, drain);
      }
      __syncwarp();
    }  // the odd CTA's MMA warp has nothing to do: its stages complete on the even CTA
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int cbase = (ew >> 2) * 128;       // this warp's 128 columns of the tile
    uint8_t* stage = sOut + ew * F_OUT_STAGE;
    const uint32_t row_off = static_cast<uint32_t>(lane) * 128;
    const uint32_t leader_tempty = map_to_rank(tempty, 0);
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    for (int tile = cluster; tile < total && ok; tile += nclusters) {
      int mt, nt;
      mmrs_tile(tile, p.m_tiles, p.n_tiles, mt, nt);
      const int grow0 = mt * 256 + static_cast<int>(rank) * 128 + q * 32;
      const int grow = grow0 + lane;
      const bool valid = grow < p.m;
      const int c0 = nt * NB + cbase;                 // first output column of this warp
      const int ncols = min(128, p.n - c0);           // <= 0, 64 or 128 (n % 64 == 0)
      float sum[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) sum[i] = 0.f;
      for (int r = 0; r < p.W; ++r) {
        if (lane == 0) ok = mbar_wait_cluster(&tfull[acc], aph, ctl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tbase = tmem_base + acc * acc_cols + static_cast<uint32_t>(cbase) +
                               (static_cast<uint32_t>(q * 32) << 16);
        const float xr = valid ? __ldg(p.xs + static_cast<int64_t>(r) * p.m + grow) : 0.f;
        const float* wr = p.ws + static_cast<int64_t>(r) * p.n + c0;
#pragma unroll
        for (int g = 0; g < 128 / GW; ++g) {
          if (g * GW < ncols) {   // no scales exist past column n
            // fp32 of the rank's exact int32 sum.  Each chunk sum is an exact
            // fp32 integer below 2^24: one chunk is that value itself, two
            // give it with one fp32 add (a single rounding of the exact sum);
            // more chunks are summed in int32 and converted.
            float af[GW];
            if (nchunk <= 2) {
              uint32_t v[GW];
              tmem_ld_group<GW>(tbase + g * GW, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < GW; ++i) af[i] = __uint_as_float(v[i]);
              if (nchunk == 2) {
                tmem_ld_group<GW>(tbase + NB + g * GW, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < GW; ++i) af[i] += __uint_as_float(v[i]);
              }
            } else {
              int32_t si[GW];
#pragma unroll
              for (int i = 0; i < GW; ++i) si[i] = 0;
#pragma unroll 1
              for (int c = 0; c < nchunk; ++c) {   // exact int32 sum of the chunk sums
                uint32_t v[GW];
                tmem_ld_group<GW>(tbase + c * NB + g * GW, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < GW; ++i) si[i] += __float2int_rn(__uint_as_float(v[i]));
              }
#pragma unroll
              for (int i = 0; i < GW; ++i) af[i] = static_cast<float>(si[i]);
            }
#pragma unroll
            for (int i = 0; i < GW; i += 4) {
              const float4 w4 = __ldg(reinterpret_cast<const float4*>(wr + g * GW + i));
              float* sp = sum + g * GW + i;
              sp[0] = __fmaf_rn(xr * w4.x, af[i], sp[0]);
              sp[1] = __fmaf_rn(xr * w4.y, af[i + 1], sp[1]);
              sp[2] = __fmaf_rn(xr * w4.z, af[i + 2], sp[2]);
              sp[3] = __fmaf_rn(xr * w4.w, af[i + 3], sp[3]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&tempty[acc]);
          else mbar_arrive_remote_relaxed(leader_tempty + acc * 8);  // after tcgen05.wait::ld
        }
        if (bufs == 2) acc ^= 1;
        if (acc == 0) aph ^= 1;
      }
      if (!ok) break;
      if (grow0 < p.m) {  // rows past m fall outside the output map and are not written
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h * 64 < ncols) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const int c = h * 64 + v * 8;
              *reinterpret_cast<uint4*>(stage + row_off + ((v ^ (lane & 7)) << 4)) =
                  make_uint4(pack_bf16x2(sum[c], sum[c + 1]), pack_bf16x2(sum[c + 2], sum[c + 3]),
                             pack_bf16x2(sum[c + 4], sum[c + 5]),
                             pack_bf16x2(sum[c + 6], sum[c + 7]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOut, stage, c0 + h * 64, grow0);
              bulk_commit();
            }
            __syncwarp();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, F_TMEM_COLS);
}

template <int NB>
cudaError_t launch_fused(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tOut,
                         FParams p, cudaStream_t st) {
  using C = FCfg<NB>;
  p.n_tiles = (p.n + NB - 1) / NB;
  p.m_tiles = (p.m + 255) / 256;
  p.total = p.m_tiles * p.n_tiles;
  // Persistent grid: as many pairs as can be resident at once (a pair needs
  // two SMs of one GPC, so this can be fewer than SMs / 2).
  static PerDevice<KernelSetup> setup;
  const KernelSetup su = once_per_device(
      setup, [] { return setup_kernel(mmrs_fused_kernel<NB>, C::kSmem, C::kThreads, true); });
  if (su.err != cudaSuccess) return su.err;
  const int max_clusters = su.pair_clusters;
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  const int grid = 2 * std::min(max_clusters, std::max(p.total, 1));
  return launch_kernel(mmrs_fused_kernel<NB>, dim3(grid), dim3(C::kThreads), C::kSmem, st, 2, tA,
                       tB, tOut, p);
}

// 256-column tiles while two K chunks fit in TMEM (K <= 2048), else 128.
cudaError_t launch_mmrs_fused(const mc2_mmrs_shape_t& s, const void* x1b, const void* x2b,
                              const float* xs, const float* ws, void* out, int32_t* dev_status,
                              cudaStream_t st) {
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t rows = static_cast<uint64_t>(s.W) * s.m;
  CUtensorMap tA, tB, tOut;
  if (!encode_2d(&tA, bf, 2, x1b, s.k, rows, 64, 128) ||
      !encode_3d(&tB, bf, 2, x2b, s.n, s.k, s.W, 64, 64) ||
      !encode_2d(&tOut, bf, 2, out, s.n, s.m, 64, 32))
    return cudaErrorInvalidValue;
  FParams p;
  p.xs = xs;
  p.ws = ws;
  p.dev_status = dev_status;
  p.W = s.W;
  p.m = s.m;
  p.n = s.n;
  p.K = s.k;
  p.nchunk = (s.k / 64 + F_CHUNK_KB - 1) / F_CHUNK_KB;
  p.wait_limit_ns = wait_limit_ns();
  const cudaError_t e = p.nchunk <= 2 ? launch_fused<256>(tA, tB, tOut, p, st)
                                      : launch_fused<128>(tA, tB, tOut, p, st);
  note_launches(1);
  return e;
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
  cudaError_t e = launch_i8_to_bf16_2(x1, w + L.x1_b16, static_cast<size_t>(rows) * s->k, x2,
                                      w + L.x2_b16, static_cast<size_t>(s->W) * s->k * s->n, st);
  if (mmrs_path_override() != 1) {  // fused: one kernel after the copies
    if (e == cudaSuccess)
      e = launch_mmrs_fused(*s, w + L.x1_b16, w + L.x2_b16, x1_scale, x2_scale, out, dev_status, st);
    return e == cudaSuccess ? MC2_OK : MC2_ERR_CUDA;
  }
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
