// wgrad.cu -- the weight gradients of the block's two grouped matmuls
// ("NPU Training Operators - MC2", section "Execution path", steps 7 and 9,
// taken backwards): for every expert e and the permuted rows p of that
// expert (offsets[e] <= p < offsets[e+1]),
//
//   dW[e] = A_e^T @ B_e            A [R, M] and B [R, N] bf16, dW [E, M, N] fp32
//
// (dw2: A = probs-weighted h, B = the gathered output gradient rows;
//  dw1: A = the permuted x rows, B = dG).  The token rows are the reduction
// axis, so both operands are MN-major: a k-block is 64 consecutive rows of A
// and of B, loaded as 128-byte-swizzled [64 rows][64 columns] blocks through
// TMA.  The last k-block of an expert reaches into the next expert's rows:
// only its 16-row MMA steps with rows of the expert are issued, and the A
// rows past the expert's end inside the last step are zeroed first (zeroing
// the whole tail of B instead cost a quarter of the kernel's time).  One CTA per 128 x 256 output tile, the expert's rows in
// order, so each tile is written once (no split over K, no atomics).
//
// Warp roles: warp 0 TMA producer, warp 1 MMA issuer (all 32 lanes zero the
// ragged rows), warps 2-5 epilogue (TMEM -> fp32 -> TMA store; zero tiles of
// experts without rows).
#include <algorithm>
#include <mutex>

#include "gmm_common.cuh"

namespace mc2 {
namespace {

constexpr int WG_BM = 128;                     // output rows (M) per tile
constexpr int WG_BN = 256;                     // output columns (N) per tile
constexpr int WG_BK = 64;                      // token rows per k-block
constexpr int WG_STAGES = 4;
constexpr int WG_A_STAGE = 2 * 8192;           // two [64 rows][64 cols] blocks
constexpr int WG_B_STAGE = 4 * 8192;           // four blocks
constexpr int WG_STAGE_BYTES = WG_A_STAGE + WG_B_STAGE;
constexpr int WG_OUT_STAGE = 4096;             // per epilogue warp: 32 rows x 32 fp32
constexpr size_t WG_SMEM = 1024 + WG_STAGES * WG_STAGE_BYTES + 4 * WG_OUT_STAGE + 256;
constexpr int WG_THREADS = 6 * 32;

struct WgradParams {
  const int32_t* offsets;
  int32_t* dev_status;
  int E, M, N, mt, nt;
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ void wg_decode(int tile, const WgradParams& p, int& e, int& m, int& n) {
  const int per = p.mt * p.nt;
  e = tile / per;
  const int r = tile - e * per;
  m = r / p.nt;
  n = r - m * p.nt;
}

__global__ void __launch_bounds__(WG_THREADS, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmOut, const WgradParams p) {
  constexpr uint32_t IDESC = instr_desc(1, true, true, WG_BM, WG_BN);  // bf16, both MN-major
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + WG_STAGES * WG_A_STAGE;
  uint8_t* sOut = sB + WG_STAGES * WG_B_STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + 4 * WG_OUT_STAGE);
  uint64_t* empty = full + WG_STAGES;
  uint64_t* tfull = empty + WG_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_sh = reinterpret_cast<volatile int*>(tmem_base_sh + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < WG_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4 * 32);
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
    tmem_alloc(tmem_base_sh, 512);
    tmem_relinquish();
  }
  griddep_wait();
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_sh;
  WaitCtl ctl{abort_sh, p.wait_limit_ns, p.dev_status};
  const int total = p.E * p.mt * p.nt;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int s = 0;
    uint32_t ph = 0;
    int n_arm = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int e, m, n;
      wg_decode(tile, p, e, m, n);
      const int r0 = __ldg(p.offsets + e), r1 = __ldg(p.offsets + e + 1);
      for (int k0 = r0; k0 < r1; k0 += WG_BK) {
        if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1, ctl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], WG_STAGE_BYTES);
          tma_load_4d(sA + s * WG_A_STAGE, &tmA, &full[s], 0, k0, 2 * m, 0);
          tma_load_4d(sB + s * WG_B_STAGE, &tmB, &full[s], 0, k0, 4 * n, 0);
        }
        __syncwarp();
        ++n_arm;
        if (++s == WG_STAGES) { s = 0; ph ^= 1; }
      }
    }
    if (lane == 0) {  // every armed stage has landed before the CTA can exit
      volatile int never = 0;
      WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
      for (int st = 0; st < WG_STAGES && st < n_arm; ++st) {
        const int last = st + WG_STAGES * ((n_arm - 1 - st) / WG_STAGES);
        mbar_wait(&full[st], (last / WG_STAGES) & 1, drain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int s = 0, acc = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int e, m, n;
      wg_decode(tile, p, e, m, n);
      const int r0 = __ldg(p.offsets + e), r1 = __ldg(p.offsets + e + 1);
      if (lane == 0) ok = mbar_wait(&tempty[acc], aph ^ 1, ctl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * WG_BN;
      for (int k0 = r0; k0 < r1; k0 += WG_BK) {
        if (lane == 0) ok = mbar_wait(&full[s], ph, ctl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // The block's rows past r1 belong to the next expert.  Only the
        // 16-row MMA steps holding rows of expert e are issued, and inside
        // the last of them the A rows past r1 (both 64-column blocks, at most
        // 15 rows) are zeroed so they add nothing.
        const int rv = r1 - k0;  // rows of this block that belong to expert e
        int nk = WG_BK / 16;
        if (rv < WG_BK) {
          nk = (rv + 15) / 16;
          const int nz = nk * 16 - rv;  // rows [rv, nk * 16) of A
          uint8_t* a = sA + s * WG_A_STAGE;
          for (int c = lane; c < 2 * nz * 8; c += 32) {
            const int blk = c / (nz * 8);
            const int rem = c - blk * nz * 8;
            *reinterpret_cast<uint4*>(a + blk * 8192 + (rv + rem / 8) * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a_base = smem_u32(sA + s * WG_A_STAGE);
          const uint32_t b_base = smem_u32(sB + s * WG_B_STAGE);
          for (int kk = 0; kk < nk; ++kk) {
            const uint64_t adesc = smem_desc_sw128(a_base + kk * 2048, 8192, 1024);
            const uint64_t bdesc = smem_desc_sw128(b_base + kk * 2048, 8192, 1024);
            umma<0>(d_tmem, adesc, bdesc, IDESC, (k0 != r0 || kk != 0) ? 1u : 0u);
          }
          umma_commit(&empty[s]);
        }
        __syncwarp();
        if (++s == WG_STAGES) { s = 0; ph ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(&tfull[acc]);  // with no MMA issued it arrives at once
      __syncwarp();
      acc ^= 1;
      if (acc == 0) aph ^= 1;
    }
    if (lane == 0) {
      umma_commit(mma_done);
      volatile int never = 0;
      WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
      mbar_wait(mma_done, 0, drain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    uint8_t* stage = sOut + q * WG_OUT_STAGE;
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, m, n;
      wg_decode(tile, p, e, m, n);
      const bool empty_expert = __ldg(p.offsets + e + 1) == __ldg(p.offsets + e);
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&tfull[acc], aph, ctl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * WG_BN + (static_cast<uint32_t>(q * 32) << 16);
      const int mrow0 = m * WG_BM + q * 32;  // first output row (of M) of this warp
      if (mrow0 < p.M) {
        const int grow0 = e * p.M + mrow0;
#pragma unroll 1
        for (int gi = 0; gi < WG_BN / 32; ++gi) {
          const int col0 = n * WG_BN + gi * 32;
          if (col0 >= p.N) break;
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          uint32_t v[32];
          if (!empty_expert) {
            tmem_ld32(tbase + gi * 32, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
#pragma unroll
          for (int w = 0; w < 8; ++w)
            *reinterpret_cast<uint4*>(stage + lane * 128 + ((w ^ (lane & 7)) << 4)) =
                make_uint4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmOut, stage, col0, grow0);
            bulk_commit();
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) aph ^= 1;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

}  // namespace

// dW [E, M, N] fp32 = per expert A_e^T @ B_e, A [R, M], B [R, N] bf16 rows in
// expert-major order (offsets [E+1]).  M and N multiples of 64.
cudaError_t launch_wgrad(const void* a, const void* b, const int32_t* offsets, int64_t R, int E,
                         int M, int N, float* dw, int32_t* dev_status, cudaStream_t st) {
  if (E == 0) return cudaSuccess;
  CUtensorMap tA, tB, tOut;
  const uint64_t rows = static_cast<uint64_t>(std::max<int64_t>(R, 1));
  // [R, M] as (64 columns, R rows, M/64 blocks, 1): box (64, 64, 2, 1) = one k-block of A
  bool ok = encode_b_blocked(&tA, a, rows, M, 1, 1, WG_BK, 2, 1) &&
            encode_b_blocked(&tB, b, rows, N, 1, 1, WG_BK, 4, 1) &&
            encode_2d(&tOut, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dw, N,
                      static_cast<uint64_t>(E) * M, 32, 32);
  if (!ok) return cudaErrorInvalidValue;
  WgradParams p;
  p.offsets = offsets;
  p.dev_status = dev_status;
  p.E = E;
  p.M = M;
  p.N = N;
  p.mt = (M + WG_BM - 1) / WG_BM;
  p.nt = (N + WG_BN - 1) / WG_BN;
  p.wait_limit_ns = wait_limit_ns();
  static PerDevice<KernelSetup> setup;
  const KernelSetup su =
      once_per_device(setup, [] { return setup_kernel(wgrad_kernel, WG_SMEM, WG_THREADS, false); });
  if (su.err != cudaSuccess) return su.err;
  const int64_t tiles = static_cast<int64_t>(E) * p.mt * p.nt;
  const int grid = static_cast<int>(std::min<int64_t>(num_sms(), tiles));
  const cudaError_t e = launch_kernel(wgrad_kernel, dim3(grid), dim3(WG_THREADS), WG_SMEM, st, 1,
                                      tA, tB, tOut, p);
  note_launches(1);
  return e;
}

}  // namespace mc2
