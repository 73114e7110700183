// gmm.cu -- the two grouped matmuls of the block on 5th-generation tensor
// cores, with the data movement of the expert-parallel exchange folded in
// ("NPU Training Operators - MC2", sections "Background constraints" and
// "Execution path", steps 6-10):
//
//   fc1 (dispatch segment):  h[p, :] = SwiGLU( x[permute_src[p] / k, :] @ w1[e] )
//        the permute is a row gather straight into the swizzled A tile
//        (cp.async by four gather warps); SwiGLU runs on the fp32
//        accumulator in TMEM; h tiles leave through TMA stores.
//   fc2 (combine segment):   y[p, :] = h[p, :] @ w2[e]   (expert-major rows)
//        stored as fp16 times a power-of-two factor per 64 columns, then
//        combine_kernel: out[t] = sum_j probs[t, j] * y[unpermute_dst[t*k+j]]
//        in ascending j -- every y row is written once, so the sum has a
//        fixed order and the result is bitwise reproducible.
//   Two more fc1 modes: MODE_FC1_ROWS takes already permuted rows through
//   TMA (the non-fused baseline path); MODE_FC1_PRE writes the
//   pre-activation gate | up rows instead of h (the backward's G).  The fc2
//   kernel also serves the backward's two dgrads (on transposed weights).
//
// One persistent kernel per segment, one CTA per SM:
//   warp 0      TMA producer of the B (weight) tiles (and of fc2's A tiles)
//   warp 1      TMEM allocator and tcgen05.mma issuer (one lane)
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, math, swizzled smem
//               staging, TMA store of 32-row boxes
//   warps 6..9  fc1 only: gather of the A rows (cp.async, 16 B per lane)
// A 4-stage ring of 48 KB stages (128-byte swizzle) feeds 128x256 UMMA tiles;
// two 256-column fp32 accumulators in TMEM (all 512 columns) let the epilogue
// of tile i overlap the mainloop of tile i+1.  Tiles are (expert, n-tile,
// m-tile) triples over a per-expert tile prefix that each CTA builds from
// `offsets`, so empty experts cost nothing and skewed ones just own more
// tiles; CTAs take tiles round-robin, and the m-tiles of one (expert,
// n-tile) are adjacent so concurrently running CTAs share its weight tile in L2.
//
// Why a cp.async gather and not TMA tile::gather4: on GB300 the gather4
// version of fc1 took 537 us on the 4096-token workload against 237 us for
// an early form of this one (190 us now; 175 us on pre-permuted rows, which
// cost a 41 us permute pass first), with bit-identical h.
//
// Below the single-CTA kernel: a CTA-pair variant (tcgen05 cta_group::2,
// 256-row tiles), used for fc2 when experts average >= 256 rows.
#include <algorithm>

#include "gmm_common.cuh"

namespace mc2 {

template <int MODE>
constexpr bool kIsFc2 = MODE == MODE_FC2 || MODE == MODE_FC2C;

// Warps 6..9: fc1's row gather, or fc2's combine warps when the combine is fused.
template <int MODE>
struct Roles {
  static constexpr int kGatherWarps =
      MODE == MODE_FC1 || MODE == MODE_FC1_PRE || MODE == MODE_FC2C ? 4 : 0;
  static constexpr int kThreads = (6 + kGatherWarps) * 32;
};

constexpr size_t SMEM_BYTES_FIXED = 1024 + STAGES * STAGE_BYTES + 4 * OUT_STAGE + 256;
constexpr int NB1 = BN / 64;  // 64-column blocks of a bf16 B tile

// ----------------------------------------------------------------------------
// The weighted combine fused into fc2 (MODE_FC2C; selected by
// mc2_set_combine_path(1), the separate combine_kernel is the default).
//
// out[t, :] = sum_j probs[t, j] * y(t, j) needs the k fc2 rows of token t,
// which different tiles (different experts) produce on different SMs.  Each
// (token, BN-column tile) has an arrival counter in the workspace, set by
// combine_prep_kernel to k minus the token's valid slots.  An epilogue warp,
// once the stores of its 32 rows of a tile have completed (checked one tile
// later, so the wait costs nothing), hands the row range through a
// shared-memory queue to its paired combine warp (warps 6..9).  The combine
// warp publishes the rows at GPU scope and adds one arrival per row; the
// row that brings a counter to k is its token's last.  It sums up to
// COMBINE_LOCAL_TOKENS such tokens per row range itself -- 8 columns per
// lane, all k rows of two tokens loaded before the first add -- and appends
// the rest to a list that combine_deferred_kernel sums after fc2.  Every sum
// uses combine_kernel's arithmetic and slot order, so the output is bitwise
// the same as the separate pass.
//
// Measured on GB300 (fc2 + combine, 4096- / 16384-token workloads): separate
// kernel 0.132 / 0.407 ms; this form 0.157 / 0.457 ms with 4 local tokens,
// 0.144 / 0.432 ms deferring all, 0.221 / 0.563 ms summing all locally.  A
// token completes only with its highest-numbered expert, so in the
// expert-major tile order most tokens complete in the last tiles, where four
// latency-bound warps per SM cannot keep up; and sums during the mainloop
// take issue slots and memory bandwidth from the GEMM.
// ----------------------------------------------------------------------------
constexpr int CQ_SLOTS = 8;
constexpr int KMAX_FUSED = 8;   // top-k handled by the fused combine

struct CombineSlot {  // rows [grow0, grow0 + wrows) of column tile n are stored; n = -1: done
  int32_t n, grow0, wrows;
};

struct CombineQueue {  // one per epilogue warp
  uint64_t full[CQ_SLOTS];
  uint64_t empty[CQ_SLOTS];
  CombineSlot slot[CQ_SLOTS];
};

constexpr int CQ_BYTES = static_cast<int>((4 * sizeof(CombineQueue) + 7) / 8 * 8);

template <int MODE>
constexpr int kQueueBytes = MODE == MODE_FC2C ? CQ_BYTES : 0;

__device__ __forceinline__ void combine_queue_init(CombineQueue* cq) {
  for (int q = 0; q < 4; ++q)
    for (int s = 0; s < CQ_SLOTS; ++s) {
      mbar_init(&cq[q].full[s], 1);
      mbar_init(&cq[q].empty[s], 1);
    }
}

// Epilogue side: rows [grow0, grow0 + wrows) of column tile n have been
// stored and lane 0 has waited for its bulk stores and fenced the async
// proxy; hand the rows to the paired combine warp.  Lane 0 only.
__device__ __forceinline__ bool combine_push(CombineQueue* q, int& qs, uint32_t& qph, int n,
                                             int grow0, int wrows, const WaitCtl& ctl) {
  if (!mbar_wait(&q->empty[qs], qph ^ 1, ctl)) return false;
  q->slot[qs] = CombineSlot{n, grow0, wrows};
  mbar_arrive(&q->full[qs]);  // release (CTA scope): the stores this warp made or waited for
  if (++qs == CQ_SLOTS) { qs = 0; qph ^= 1; }
  return true;
}

__device__ __forceinline__ void combine_add(float (&acc)[8], float pj, float f, const uint4& raw) {
  const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __half22float2(h2[i]);
    acc[2 * i] += __fmul_rn(pj, v.x * f);
    acc[2 * i + 1] += __fmul_rn(pj, v.y * f);
  }
}

struct CombineArgs {
  const __half* y;          // fc2 rows [R, H], fp16 scaled
  const float* yscale;      // [R, H/64]
  void* out;                // [T, H] bf16 or fp32
  int H, out_f32;
  int32_t nvalid;           // rows p >= nvalid belong to invalid ids
};

// Sums NJ (token, column) jobs: out[t[u], col[u] .. +8) = sum over j
// ascending of pj[u][j] * y(r[u][j]) for the valid rows r < nvalid.  A job
// with t < 0 or an inactive column is skipped.  Every load of all jobs is
// issued before the first add.
template <int NJ>
__device__ __forceinline__ void combine_jobs(const CombineArgs& a, const int (&t)[NJ],
                                             const int (&col)[NJ],
                                             const int32_t (&r)[NJ][KMAX_FUSED],
                                             const float (&pj)[NJ][KMAX_FUSED]) {
  float f[NJ][KMAX_FUSED];
  uint4 raw[NJ][KMAX_FUSED];
  const int HG = a.H / 64;
#pragma unroll
  for (int u = 0; u < NJ; ++u)
#pragma unroll
    for (int j = 0; j < KMAX_FUSED; ++j) {
      const bool ok = t[u] >= 0 && col[u] < a.H && r[u][j] < a.nvalid;
      const int64_t rr = ok ? r[u][j] : 0;
      f[u][j] = ok ? ld_cg_f32(a.yscale + rr * HG + col[u] / 64) : 0.f;
      raw[u][j] = ok ? ld_cg_u4(a.y + rr * a.H + col[u]) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
  for (int u = 0; u < NJ; ++u) {
    if (t[u] < 0 || col[u] >= a.H) continue;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX_FUSED; ++j)
      if (r[u][j] < a.nvalid) combine_add(acc, pj[u][j], f[u][j], raw[u][j]);
    const int64_t o = static_cast<int64_t>(t[u]) * a.H + col[u];
    if (a.out_f32) {
      float4* d = reinterpret_cast<float4*>(static_cast<float*>(a.out) + o);
      d[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      d[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + o) =
          make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                     pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
  }
}

// Tokens whose last row arrives while a combine warp still has a backlog are
// not summed there but appended to a list in the workspace (item = token *
// n_tiles + column tile); combine_deferred_kernel sums them after fc2 with
// the whole GPU.  A combine warp sums at most this many tokens per batch of
// stored rows itself, which keeps pace with the tiles during the mainloop;
// the burst at the end (a token completes with its highest expert, so most
// tokens complete in the last tiles of the expert-major order) is deferred.
constexpr int COMBINE_LOCAL_TOKENS = 4;

// A combine warp: takes stored row ranges from its queue until the epilogue
// warp sends n = -1 (or the CTA aborts).  For each range: publish the rows
// at GPU scope, add one arrival per row, and sum (or defer) every token whose
// last row this was.
__device__ __forceinline__ void combine_warp(const GemmParams& p, CombineQueue* q, int lane,
                                             const WaitCtl& ctl) {
  const int k = p.k;
  CombineArgs a;
  a.y = static_cast<const __half*>(p.out);
  a.yscale = p.yscale;
  a.out = p.comb_out;
  a.H = p.out_cols;
  a.out_f32 = p.out_f32;
  a.nvalid = __ldg(p.offsets + p.E);
  int qs = 0;
  uint32_t qph = 0;
  while (true) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait(&q->full[qs], qph, ctl);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    const CombineSlot sl = q->slot[qs];
    __syncwarp();
    if (lane == 0) mbar_arrive(&q->empty[qs]);
    if (++qs == CQ_SLOTS) { qs = 0; qph ^= 1; }
    if (sl.n < 0) break;
    fence_acq_rel_gpu();  // release the stored rows (observed through the queue) before arriving
    int tok = 0;
    bool last = false;
    int32_t myr[KMAX_FUSED];
    float myp[KMAX_FUSED];
    if (lane < sl.wrows) {
      tok = __ldg(p.permute_src + sl.grow0 + lane) / k;
      const int old = atomicAdd(p.ctr + static_cast<int64_t>(tok) * p.n_tiles + sl.n, 1);
#pragma unroll
      for (int j = 0; j < KMAX_FUSED; ++j) {  // this token's rows and weights, in case it is done
        myr[j] = j < k ? __ldg(p.unpermute_dst + static_cast<int64_t>(tok) * k + j) : a.nvalid;
        myp[j] = j < k ? __ldg(p.probs + static_cast<int64_t>(tok) * k + j) : 0.f;
      }
      last = old == k - 1;
    } else {
#pragma unroll
      for (int j = 0; j < KMAX_FUSED; ++j) {
        myr[j] = a.nvalid;
        myp[j] = 0.f;
      }
    }
    uint32_t mask = __ballot_sync(0xffffffffu, last);
    if (!mask) continue;
    // beyond the local budget: defer (warp-aggregated append to the list)
    uint32_t local = 0;
    for (int i = 0; i < COMBINE_LOCAL_TOKENS && (mask & ~local); ++i)
      local |= (mask & ~local) & (0u - (mask & ~local));  // lowest remaining bit
    const uint32_t defer = mask & ~local;
    if (defer) {
      int base = 0;
      if (lane == 0) base = atomicAdd(p.defer_count, __popc(defer));
      base = __shfl_sync(0xffffffffu, base, 0);
      if ((defer >> lane) & 1u)
        p.defer_items[base + __popc(defer & ((1u << lane) - 1u))] = tok * p.n_tiles + sl.n;
    }
    if (!local) continue;
    fence_acq_rel_gpu();  // acquire the tokens' other rows, released by their writers
    const int colv = sl.n * BN + 8 * lane;
    mask = local;
    while (mask) {
      const int b0 = __ffs(mask) - 1;
      mask &= mask - 1;
      const bool two = mask != 0;
      const int b1 = two ? __ffs(mask) - 1 : b0;
      if (two) mask &= mask - 1;
      int t[2] = {__shfl_sync(0xffffffffu, tok, b0), __shfl_sync(0xffffffffu, tok, b1)};
      if (!two) t[1] = -1;
      const int col[2] = {colv, colv};
      int32_t r[2][KMAX_FUSED];
      float pj[2][KMAX_FUSED];
#pragma unroll
      for (int j = 0; j < KMAX_FUSED; ++j) {
        r[0][j] = __shfl_sync(0xffffffffu, myr[j], b0);
        pj[0][j] = __shfl_sync(0xffffffffu, myp[j], b0);
        r[1][j] = __shfl_sync(0xffffffffu, myr[j], b1);
        pj[1][j] = __shfl_sync(0xffffffffu, myp[j], b1);
      }
      combine_jobs<2>(a, t, col, r, pj);
    }
  }
}

// Wait until at most `keep` of this thread's most recent bulk-store groups
// are still in flight (keep = 0..4).
__device__ __forceinline__ void bulk_wait_keep_n(int keep) {
  switch (keep) {
    case 0: bulk_wait_keep<0>(); break;
    case 1: bulk_wait_keep<1>(); break;
    case 2: bulk_wait_keep<2>(); break;
    case 3: bulk_wait_keep<3>(); break;
    default: bulk_wait_keep<4>(); break;
  }
}

template <int MODE, int ES>
__global__ void __launch_bounds__(Roles<MODE>::kThreads, 1)
    gmm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
  using TR = ElemTraits<ES>;
  constexpr int BK = TR::BK;
  constexpr int BNB = 128 / ES;              // columns per 128-byte B block
  constexpr int NB = BN / BNB;               // B blocks per stage
  constexpr int B_BLOCK = BK * 128;          // bytes per B block (BK rows x 128 B)
  constexpr int KK_B = (32 / ES) * 128;      // B bytes per UMMA K step
  constexpr bool BKM = TR::B_KMAJOR;
  constexpr uint32_t IDESC = instr_desc(TR::FMT, false, !BKM, BM, BN);
  constexpr bool GATHER = MODE == MODE_FC1 || MODE == MODE_FC1_PRE;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE;
  uint8_t* sOut = sB + STAGES * B_STAGE;
  CombineQueue* cq = reinterpret_cast<CombineQueue*>(sOut + 4 * OUT_STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + 4 * OUT_STAGE + kQueueBytes<MODE>);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_sh = reinterpret_cast<volatile int*>(tmem_base_sh + 1);
  int32_t* prefix = reinterpret_cast<int32_t*>(tmem_base_sh + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int unit = static_cast<int>(blockIdx.x);
  const int nunits = static_cast<int>(gridDim.x);
  // this CTA's rows of tile `tile`: [row0, row0 + rows)
  auto tile_at = [&](int tile, int& e, int& n, int& row0, int& rows) {
    decode_tile(tile, prefix, E, p.n_tiles, p.offsets, e, n, row0, rows);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // fc1: the TMA arm of the B tile plus one arrival per gather thread
      mbar_init(&full[s], GATHER ? 1 + 32 * Roles<MODE>::kGatherWarps : 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4 * 32);
    }
    mbar_init(mma_done, 1);
    if constexpr (MODE == MODE_FC2C) combine_queue_init(cq);
    *abort_sh = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    if (!GATHER) tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_sh, TMEM_COLS);
    tmem_relinquish();
  }
  // everything above touches only shared memory, TMEM and the parameter
  // space, so it overlaps the end of the previous kernel in the stream
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 2) {  // per-expert tile prefix: ceil(rows_e / BM) * n_tiles
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int t = 0;
      if (e < E) {
        const int rows = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
        t = ((rows + BM - 1) / BM) * p.n_tiles;
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      if (e < E) prefix[e + 1] = run + t;
      run += __shfl_sync(0xffffffffu, t, 31);
    }
    if (lane == 0) prefix[0] = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_sh;
  const int total = prefix[E];
  WaitCtl ctl{abort_sh, p.wait_limit_ns, p.dev_status};
  const int kblocks = p.K / BK;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int s = 0;
    uint32_t ph = 0;
    int n_arm = 0;
    bool ok = true;
    for (int tile = unit; tile < total && ok; tile += nunits) {
      int e, n, row0, rows;
      tile_at(tile, e, n, row0, rows);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1, ctl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], GATHER ? B_STAGE : STAGE_BYTES);
          uint8_t* b_dst = sB + s * B_STAGE;
          const int k0 = kb * BK;
          if (!GATHER) tma_load_2d(sA + s * A_STAGE, &tmA, &full[s], k0, row0);
          if constexpr (BKM) {
            // K-major B: N rows of 128 bytes of K; fc1 loads the gate rows
            // and the up rows of the same output columns as two boxes
            if (!kIsFc2<MODE>) {
              tma_load_3d(b_dst, &tmB, &full[s], k0, n * (BN / 2), e);
              tma_load_3d(b_dst + (BN / 2) * 128, &tmB, &full[s], k0, p.I + n * (BN / 2), e);
            } else {
              tma_load_3d(b_dst, &tmB, &full[s], k0, n * BN, e);
            }
          } else {
            // all NB 64-column blocks in one box: fc1 takes the gate and the
            // up blocks of the same output columns, fc2 NB adjacent blocks
            if (!kIsFc2<MODE>)
              tma_load_5d(b_dst, &tmB, &full[s], 0, k0, n * (NB / 2), 0, e);
            else
              tma_load_4d(b_dst, &tmB, &full[s], 0, k0, n * NB, e);
          }
        }
        __syncwarp();
        ++n_arm;
        if (++s == STAGES) { s = 0; ph ^= 1; }
      }
    }
    // Let every armed stage land before the CTA can exit (bounded).
    if (lane == 0) {
      volatile int never = 0;
      WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
      for (int st = 0; st < STAGES && st < n_arm; ++st) {
        const int last = st + STAGES * ((n_arm - 1 - st) / STAGES);
        mbar_wait(&full[st], (last / STAGES) & 1, drain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int s = 0;
    uint32_t ph = 0;
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    for (int tile = unit; tile < total && ok; tile += nunits) {
      if (lane == 0) ok = mbar_wait(&tempty[acc], aph ^ 1, ctl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (lane == 0) {
          ok = mbar_wait(&full[s], ph, ctl);
          if (GATHER && ok) fence_proxy_async_smem();  // gathered rows -> async proxy
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a_base = smem_u32(sA + s * A_STAGE);
          const uint32_t b_base = smem_u32(sB + s * B_STAGE);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = BKM ? smem_desc_sw128(b_base + kk * 32, 16, 1024)
                                       : smem_desc_sw128(b_base + kk * KK_B, B_BLOCK, 1024);
            umma<TR::KIND>(d_tmem, adesc, bdesc, IDESC, (kb | kk) != 0);
          }
          umma_commit(&empty[s]);
        }
        __syncwarp();
        if (++s == STAGES) { s = 0; ph ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(&tfull[acc]);
      __syncwarp();
      acc ^= 1;
      if (acc == 0) aph ^= 1;
    }
    if (lane == 0) {  // every issued MMA has finished reading smem / writing TMEM
      umma_commit(mma_done);
      volatile int never = 0;
      WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
      mbar_wait(mma_done, 0, drain);
    }
    __syncwarp();
  } else if (MODE == MODE_FC2C && warp >= 6) {
    // ------------------------------------------------------------ fused combine
    combine_warp(p, cq + (warp - 6), lane, ctl);
  } else if (warp >= 6) {
    // ------------------------------------------------------------ fc1 row gather
    // Thread t copies 16-byte chunk (t % 8) of rows t/8 + 16*i, i = 0..7, of
    // the 128-row A tile: 8 lanes cover one 128-byte row segment, so each
    // warp instruction reads four whole rows.  The chunk lands at its 128B
    // swizzle position.  Each thread's copies into a stage arrive on full[s]
    // when they land (cp.async.mbarrier.arrive), so the gather runs as far
    // ahead as the ring has free stages; the MMA thread fences the async
    // proxy after its wait.
    const int t = threadIdx.x - 6 * 32;
    const int chunk = t & 7, rsub = t >> 3;
    const char* xg = static_cast<const char*>(p.a_ptr);
    const int64_t row_bytes = static_cast<int64_t>(p.K) * ES;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tile = unit; tile < total && ok; tile += nunits) {
      int e, n, row0, rows;
      tile_at(tile, e, n, row0, rows);
      const int tok0 = __ldg(p.permute_src + row0) / p.k;  // tail rows repeat a valid row
      const char* src[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = rsub + 16 * i;
        const int tok = r < rows ? __ldg(p.permute_src + row0 + r) / p.k : tok0;
        src[i] = xg + tok * row_bytes + chunk * 16;
      }
      for (int kb = 0; kb < kblocks; ++kb) {
        if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1, ctl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t a_dst = smem_u32(sA + s * A_STAGE);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = rsub + 16 * i;
          cp_async16(a_dst + r * 128 + ((chunk ^ (r & 7)) << 4), src[i] + kb * 128);
        }
        cp_async_mbar_arrive_noinc(&full[s]);
        if (++s == STAGES) { s = 0; ph ^= 1; }
      }
    }
    cp_async_wait<0>();
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp q owns accumulator rows 32q..32q+31 (TMEM lane quarter q).  Each
    // 128-byte column group of its rows is staged in swizzled smem and
    // written by one TMA store of a 32-row box; a warp whose rows run past
    // the end of the expert stores its valid rows directly instead.
    const int q = warp & 3;
    uint8_t* stage = sOut + q * OUT_STAGE;
    const uint32_t row_off = static_cast<uint32_t>(lane) * 128;
    int acc = 0;
    uint32_t aph = 0;
    // fused combine: the previous tile's rows wait here until their stores complete
    int pend_grow0 = 0, pend_wrows = 0, pend_n = 0, qs = 0;
    uint32_t qph = 0;
    for (int tile = unit; tile < total; tile += nunits) {
      int e, n, row0, rows;
      tile_at(tile, e, n, row0, rows);
      int ngroups_tma = 0;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&tfull[acc], aph, ctl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
      const int wrows = min(32, rows - q * 32);       // valid rows of this warp
      const int grow0 = row0 + q * 32;                 // first global row of this warp
      if (wrows > 0) {
        constexpr int GROUP_COLS = 128 / (!kIsFc2<MODE> ? ES : 2);  // output cols per 128 B
        constexpr int NGROUPS = (!kIsFc2<MODE> ? BN / 2 : BN) / GROUP_COLS;
#pragma unroll 1
        for (int gi = 0; gi < NGROUPS; ++gi) {
          const int col0 = n * (!kIsFc2<MODE> ? BN / 2 : BN) + gi * GROUP_COLS;
          if (col0 >= p.out_cols) break;
          if constexpr (MODE == MODE_FC1_PRE) {
            // the previous store out of this warp's staging buffer has read it
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            // gate then up columns of G [R, 2I], bf16, as they leave the MMA
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {
              if (part) {
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
              }
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                uint32_t v[32];
                tmem_ld32(tbase + part * (BN / 2) + gi * 64 + half * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                  const int ch = half * 4 + w;
                  *reinterpret_cast<uint4*>(stage + row_off + ((ch ^ (lane & 7)) << 4)) =
                      make_uint4(pack_bf16x2(__uint_as_float(v[8 * w]), __uint_as_float(v[8 * w + 1])),
                                 pack_bf16x2(__uint_as_float(v[8 * w + 2]), __uint_as_float(v[8 * w + 3])),
                                 pack_bf16x2(__uint_as_float(v[8 * w + 4]), __uint_as_float(v[8 * w + 5])),
                                 pack_bf16x2(__uint_as_float(v[8 * w + 6]), __uint_as_float(v[8 * w + 7])));
                }
              }
              const int gcol = part * p.out_cols + col0;
              if (wrows == 32) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  tma_store_2d(&tmOut, stage, gcol, grow0);
                  bulk_commit();
                }
              } else if (lane < wrows) {
                uint4* dst = reinterpret_cast<uint4*>(
                    static_cast<__nv_bfloat16*>(p.out) +
                    static_cast<int64_t>(grow0 + lane) * 2 * p.out_cols + gcol);
#pragma unroll
                for (int w = 0; w < 8; ++w)
                  dst[w] = *reinterpret_cast<const uint4*>(stage + row_off + ((w ^ (lane & 7)) << 4));
              }
              __syncwarp();
            }
            continue;
          }
          if (!kIsFc2<MODE> && ES == 2) {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              uint32_t g[32], u[32];
              const int c = gi * 64 + half * 32;
              tmem_ld32(tbase + c, g);
              tmem_ld32(tbase + BN / 2 + c, u);
              tmem_ld_wait();
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                pk[i] = pack_bf16x2(silu_f(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]),
                                    silu_f(__uint_as_float(g[2 * i + 1])) *
                                        __uint_as_float(u[2 * i + 1]));
              if (half == 0) {  // the previous store out of the staging buffer has read it
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
              }
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const int ch = half * 4 + v;
                *reinterpret_cast<uint4*>(stage + row_off + ((ch ^ (lane & 7)) << 4)) =
                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
              }
            }
          } else if (kIsFc2<MODE>) {  // y as fp16 with a power-of-two scale per 64 columns
            uint32_t a[32], b2[32], pk[32];
            tmem_ld32(tbase + gi * 64, a);
            tmem_ld32(tbase + gi * 64 + 32, b2);
            tmem_ld_wait();
            const float inv = pack_y16(a, b2, pk);
            if (lane < wrows)
              p.yscale[static_cast<int64_t>(grow0 + lane) * (p.out_cols / 64) + col0 / 64] = inv;
            if (lane == 0) bulk_wait_read_all();  // the previous store has read the staging buffer
            __syncwarp();
#pragma unroll
            for (int v = 0; v < 8; ++v)
              *reinterpret_cast<uint4*>(stage + row_off + ((v ^ (lane & 7)) << 4)) =
                  make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          } else {
            uint32_t v32[32];
            if (!kIsFc2<MODE>) {  // fp32 h, tf32-rounded for the fc2 tensor-core pass
              uint32_t g[32];
              tmem_ld32(tbase + gi * 32, g);
              tmem_ld32(tbase + BN / 2 + gi * 32, v32);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                v32[i] = __float_as_uint(
                    round_tf32(silu_f(__uint_as_float(g[i])) * __uint_as_float(v32[i])));
            } else {
              tmem_ld32(tbase + gi * 32, v32);
              tmem_ld_wait();
            }
            if (lane == 0) bulk_wait_read_all();  // the previous store has read the staging buffer
            __syncwarp();
#pragma unroll
            for (int v = 0; v < 8; ++v)
              *reinterpret_cast<uint4*>(stage + row_off + ((v ^ (lane & 7)) << 4)) =
                  make_uint4(v32[4 * v], v32[4 * v + 1], v32[4 * v + 2], v32[4 * v + 3]);
          }
          if (wrows == 32) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOut, stage, col0, grow0);
              bulk_commit();
            }
            ++ngroups_tma;
          } else if (lane < wrows) {  // tail rows: plain stores of this lane's row
            char* dst = static_cast<char*>(p.out) +
                        (static_cast<int64_t>(grow0 + lane) * p.out_cols + col0) *
                            (!kIsFc2<MODE> ? ES : 2);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<uint4*>(dst)[v] =
                  *reinterpret_cast<const uint4*>(stage + row_off + ((v ^ (lane & 7)) << 4));
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) aph ^= 1;
      if constexpr (MODE == MODE_FC2C) {
        if (pend_wrows > 0) {
          bool pushed = true;
          if (lane == 0) {  // the previous tile's stores; this tile's may stay in flight
            bulk_wait_keep_n(ngroups_tma);
            fence_proxy_async_global();
            pushed = combine_push(cq + q, qs, qph, pend_n, pend_grow0, pend_wrows, ctl);
          }
          if (!__shfl_sync(0xffffffffu, pushed, 0)) break;
        }
        pend_grow0 = grow0;
        pend_wrows = wrows > 0 ? wrows : 0;
        pend_n = n;
      }
    }
    if (lane == 0) bulk_wait_all();
    if constexpr (MODE == MODE_FC2C) {
      if (lane == 0 && *abort_sh == 0) {
        fence_proxy_async_global();
        bool ok = true;
        if (pend_wrows > 0) ok = combine_push(cq + q, qs, qph, pend_n, pend_grow0, pend_wrows, ctl);
        if (ok) combine_push(cq + q, qs, qph, -1, 0, 0, ctl);  // no more work
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ----------------------------------------------------------------------------
// CTA-pair variant: one 256x256 UMMA tile per cluster of two CTAs
// (tcgen05 cta_group::2).  Each CTA owns 128 rows of A and 128 columns of B
// -- fc1: the even CTA the gate half, the odd CTA the up half of the same 128
// output columns -- so each SM streams 32 KB per k-block instead of 48 KB,
// and six stages fit.  The even CTA issues the MMAs and commits to barriers
// in both CTAs.  With TMA-loaded operands (fc2, fc1 on permuted rows) the odd
// CTA's copies complete on the even CTA's stage barrier (pair form of the
// copy, which names a barrier in either CTA of the pair); with gathered rows
// (cp.async, local barriers only) the odd CTA's idle MMA warp relays "stage s
// landed here" to the even CTA.  Each CTA's TMEM holds all 256 accumulator columns of its 128
// rows, so the epilogue is the single-CTA one; two accumulators in TMEM let
// the epilogue of tile i overlap the mainloop of tile i+1.
// ----------------------------------------------------------------------------
constexpr int P_STAGES = 6;
constexpr int P_B_STAGE = 16384;                 // (128/es) K rows x 128 columns x es
constexpr int P_STAGE_BYTES = A_STAGE + P_B_STAGE;
constexpr int P_TMEM_COLS = 512;                 // two 256-column fp32 accumulators
constexpr size_t P_SMEM_BYTES_FIXED = 1024 + P_STAGES * P_STAGE_BYTES + 4 * OUT_STAGE + 512;

template <int MODE, int ES>
__global__ void __launch_bounds__(Roles<MODE>::kThreads, 1)
    gmm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
  using TR = ElemTraits<ES>;
  constexpr int BK = TR::BK;
  constexpr int BNB = 128 / ES;              // columns per 128-byte B block
  constexpr int NBH = (BN / 2) / BNB;        // B blocks per CTA per stage
  constexpr int B_BLOCK = BK * 128;
  constexpr int KK_B = (32 / ES) * 128;
  constexpr bool BKM = TR::B_KMAJOR;
  constexpr uint32_t IDESC = instr_desc(TR::FMT, false, !BKM, 2 * BM, BN);
  constexpr bool GATHER = MODE == MODE_FC1 || MODE == MODE_FC1_PRE;
  // TMA-only modes: the odd CTA's loads complete on the even CTA's full[s]
  // (pair form of the copy); gathering modes relay the odd CTA's stages.
  constexpr bool DIRECT = !GATHER;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + P_STAGES * A_STAGE;
  uint8_t* sOut = sB + P_STAGES * P_B_STAGE;
  CombineQueue* cq = reinterpret_cast<CombineQueue*>(sOut + 4 * OUT_STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + 4 * OUT_STAGE + kQueueBytes<MODE>);
  uint64_t* pfull = full + P_STAGES;       // even CTA: the odd CTA's stage landed
  uint64_t* empty = pfull + P_STAGES;
  uint64_t* tfull = empty + P_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_sh = reinterpret_cast<volatile int*>(tmem_base_sh + 1);
  int32_t* prefix = reinterpret_cast<int32_t*>(tmem_base_sh + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(&full[s], GATHER ? 1 + 32 * Roles<MODE>::kGatherWarps : 1);
      mbar_init(&pfull[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * 4);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(mma_done, 1);
    if constexpr (MODE == MODE_FC2C) combine_queue_init(cq);
    *abort_sh = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    if (!GATHER) tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_base_sh, P_TMEM_COLS);
    tmem_relinquish_pair();
  }
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 2) {  // per-expert tile prefix: ceil(rows_e / 256) * n_tiles
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int t = 0;
      if (e < E) {
        const int rows = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
        t = ((rows + 2 * BM - 1) / (2 * BM)) * p.n_tiles;
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      if (e < E) prefix[e + 1] = run + t;
      run += __shfl_sync(0xffffffffu, t, 31);
    }
    if (lane == 0) prefix[0] = 0;
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_sh;
  // Both CTAs of the pair must hold the same TMEM address: the MMA writes the
  // accumulator at one address in both.  Anything else aborts the kernel.
  const uint32_t peer_base = ld_shared_cluster_u32(map_to_rank(tmem_base_sh, rank ^ 1u));
  int total = prefix[E];
  if (peer_base != tmem_base) {
    if (threadIdx.x == 0 && p.dev_status) atomicOr(p.dev_status, 0x4);
    total = 0;
  }
  WaitCtl ctl{abort_sh, p.wait_limit_ns, p.dev_status};
  const int kblocks = p.K / BK;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint32_t leader_full = map_to_rank(full, 0);
    int s = 0;
    uint32_t ph = 0;
    int n_arm = 0;
    bool ok = true;
    for (int tile = cluster; tile < total && ok; tile += nclusters) {
      int e, n, prow0, prows;
      decode_tile(tile, prefix, E, p.n_tiles, p.offsets, e, n, prow0, prows);
      (void)prows;
      // decode_tile works in units of BM rows; a pair tile spans 2*BM rows
      const int local = tile - prefix[e];
      const int m_pairs = (prefix[e + 1] - prefix[e]) / p.n_tiles;
      const int mp = local - (local / m_pairs) * m_pairs;
      const int row0 = __ldg(p.offsets + e) + mp * 2 * BM + static_cast<int>(rank) * BM;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (lane == 0) ok = mbar_wait_cluster(&empty[s], ph ^ 1, ctl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          uint8_t* b_dst = sB + s * P_B_STAGE;
          const int k0 = kb * BK;
          // this CTA's 128 columns of B: fc1 gate (even) or up (odd) half;
          // fc2 the first or second 128 of the 256-column tile
          const int nbase = !kIsFc2<MODE> ? static_cast<int>(rank) * p.I + n * (BN / 2)
                                             : n * BN + static_cast<int>(rank) * (BN / 2);
          if (DIRECT && !leader) {
            const uint32_t bar = leader_full + s * 8;
            tma_load_2d_pair(sA + s * A_STAGE, &tmA, bar, k0, row0);
            if constexpr (BKM) {
              tma_load_3d_pair(b_dst, &tmB, bar, k0, nbase, e);
            } else {
              if (!kIsFc2<MODE>)
                tma_load_5d_pair(b_dst, &tmB, bar, 0, k0, n * NBH, static_cast<int>(rank), e);
              else
                tma_load_4d_pair(b_dst, &tmB, bar, 0, k0, nbase / BNB, e);
            }
          } else {
            mbar_arrive_expect_tx(&full[s], GATHER ? P_B_STAGE : 2 * P_STAGE_BYTES);
            if (!GATHER) tma_load_2d(sA + s * A_STAGE, &tmA, &full[s], k0, row0);
            if constexpr (BKM) {
              tma_load_3d(b_dst, &tmB, &full[s], k0, nbase, e);
            } else {
              if (!kIsFc2<MODE>)
                tma_load_5d(b_dst, &tmB, &full[s], 0, k0, n * NBH, static_cast<int>(rank), e);
              else
                tma_load_4d(b_dst, &tmB, &full[s], 0, k0, nbase / BNB, e);
            }
          }
        }
        __syncwarp();
        ++n_arm;
        if (++s == P_STAGES) { s = 0; ph ^= 1; }
      }
    }
    if (lane == 0) {  // every armed stage has landed and every commit to it has arrived
      volatile int never = 0;
      WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
      for (int st = 0; st < P_STAGES && st < n_arm; ++st) {
        const int last = st + P_STAGES * ((n_arm - 1 - st) / P_STAGES);
        if (!DIRECT || leader) mbar_wait_cluster(&full[st], (last / P_STAGES) & 1, drain);
        mbar_wait_cluster(&empty[st], (last / P_STAGES) & 1, drain);
      }
    }
  } else if (warp == 1) {
    if (leader) {
      // ---------------------------------------------------------- MMA issuer
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int tile = cluster; tile < total && ok; tile += nclusters) {
        if (lane == 0) ok = mbar_wait_cluster(&tempty[acc], aph ^ 1, ctl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (lane == 0) {
            ok = mbar_wait_cluster(&full[s], ph, ctl);
            if (ok && !DIRECT) ok = mbar_wait_cluster(&pfull[s], ph, ctl);
            if (GATHER && ok) fence_proxy_async_smem();  // gathered rows -> async proxy
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a_base = smem_u32(sA + s * A_STAGE);
            const uint32_t b_base = smem_u32(sB + s * P_B_STAGE);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
              const uint64_t bdesc = BKM ? smem_desc_sw128(b_base + kk * 32, 16, 1024)
                                         : smem_desc_sw128(b_base + kk * KK_B, B_BLOCK, 1024);
              umma_pair<TR::KIND>(d_tmem, adesc, bdesc, IDESC, (kb | kk) != 0);
            }
            umma_commit_pair(&empty[s], 0x3);
          }
          __syncwarp();
          if (++s == P_STAGES) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        if (lane == 0) umma_commit_pair(&tfull[acc], 0x3);
        __syncwarp();
        acc ^= 1;
        if (acc == 0) aph ^= 1;
      }
      if (lane == 0) {
        umma_commit_pair(mma_done, 0x1);
        volatile int never = 0;
        WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
        mbar_wait_cluster(mma_done, 0, drain);
      }
      __syncwarp();
    } else if (!DIRECT) {
      // ---------------------------------------------------------- relay (odd CTA)
      const uint32_t leader_pfull = map_to_rank(pfull, 0);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = cluster; tile < total && ok; tile += nclusters) {
        for (int kb = 0; kb < kblocks; ++kb) {
          if (lane == 0) {
            ok = mbar_wait(&full[s], ph, ctl);
            if (GATHER && ok) fence_proxy_async_smem();  // gathered rows -> async proxy
            if (ok) mbar_arrive_remote_relaxed(leader_pfull + s * 8);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (++s == P_STAGES) { s = 0; ph ^= 1; }
        }
      }
    }
  } else if (MODE == MODE_FC2C && warp >= 6) {
    // ------------------------------------------------------------ fused combine
    combine_warp(p, cq + (warp - 6), lane, ctl);
  } else if (warp >= 6) {
    // ------------------------------------------------------------ fc1 row gather
    const int t = threadIdx.x - 6 * 32;
    const int chunk = t & 7, rsub = t >> 3;
    const char* xg = static_cast<const char*>(p.a_ptr);
    const int64_t row_bytes = static_cast<int64_t>(p.K) * ES;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tile = cluster; tile < total && ok; tile += nclusters) {
      int e, n, prow0, prows;
      decode_tile(tile, prefix, E, p.n_tiles, p.offsets, e, n, prow0, prows);
      const int local = tile - prefix[e];
      const int m_pairs = (prefix[e + 1] - prefix[e]) / p.n_tiles;
      const int mp = local - (local / m_pairs) * m_pairs;
      const int pair0 = __ldg(p.offsets + e) + mp * 2 * BM;
      const int row0 = pair0 + static_cast<int>(rank) * BM;
      const int rows = __ldg(p.offsets + e + 1) - row0;       // may be <= 0 for the odd CTA
      const int tok0 = __ldg(p.permute_src + pair0) / p.k;    // a valid row for padding
      const char* src[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = rsub + 16 * i;
        const int tok = r < rows ? __ldg(p.permute_src + row0 + r) / p.k : tok0;
        src[i] = xg + tok * row_bytes + chunk * 16;
      }
      for (int kb = 0; kb < kblocks; ++kb) {
        if (lane == 0) ok = mbar_wait_cluster(&empty[s], ph ^ 1, ctl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t a_dst = smem_u32(sA + s * A_STAGE);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = rsub + 16 * i;
          cp_async16(a_dst + r * 128 + ((chunk ^ (r & 7)) << 4), src[i] + kb * 128);
        }
        cp_async_mbar_arrive_noinc(&full[s]);
        if (++s == P_STAGES) { s = 0; ph ^= 1; }
      }
    }
    cp_async_wait<0>();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    uint8_t* stage = sOut + q * OUT_STAGE;
    const uint32_t row_off = static_cast<uint32_t>(lane) * 128;
    const uint32_t leader_tempty = map_to_rank(tempty, 0);
    int acc = 0;
    uint32_t aph = 0;
    // fused combine: the previous tile's rows wait here until their stores complete
    int pend_grow0 = 0, pend_wrows = 0, pend_n = 0, qs = 0;
    uint32_t qph = 0;
    for (int tile = cluster; tile < total; tile += nclusters) {
      int e, n, prow0, prows;
      decode_tile(tile, prefix, E, p.n_tiles, p.offsets, e, n, prow0, prows);
      int ngroups_tma = 0;
      const int local = tile - prefix[e];
      const int m_pairs = (prefix[e + 1] - prefix[e]) / p.n_tiles;
      const int mp = local - (local / m_pairs) * m_pairs;
      const int row0 = __ldg(p.offsets + e) + mp * 2 * BM + static_cast<int>(rank) * BM;
      const int rows = __ldg(p.offsets + e + 1) - row0;
      bool ok = true;
      if (lane == 0) ok = mbar_wait_cluster(&tfull[acc], aph, ctl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
      const int wrows = min(32, rows - q * 32);
      const int grow0 = row0 + q * 32;
      if (wrows > 0) {
        constexpr int GROUP_COLS = 128 / (!kIsFc2<MODE> ? ES : 2);
        constexpr int NGROUPS = (!kIsFc2<MODE> ? BN / 2 : BN) / GROUP_COLS;
#pragma unroll 1
        for (int gi = 0; gi < NGROUPS; ++gi) {
          const int col0 = n * (!kIsFc2<MODE> ? BN / 2 : BN) + gi * GROUP_COLS;
          if (col0 >= p.out_cols) break;
          if (!kIsFc2<MODE> && ES == 2) {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              uint32_t g[32], u[32];
              const int c = gi * 64 + half * 32;
              tmem_ld32(tbase + c, g);
              tmem_ld32(tbase + BN / 2 + c, u);
              tmem_ld_wait();
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                pk[i] = pack_bf16x2(silu_f(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]),
                                    silu_f(__uint_as_float(g[2 * i + 1])) *
                                        __uint_as_float(u[2 * i + 1]));
              if (half == 0) {  // the previous store out of the staging buffer has read it
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
              }
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const int ch = half * 4 + v;
                *reinterpret_cast<uint4*>(stage + row_off + ((ch ^ (lane & 7)) << 4)) =
                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
              }
            }
          } else if (kIsFc2<MODE>) {  // y as fp16 with a power-of-two scale per 64 columns
            uint32_t a[32], b2[32], pk[32];
            tmem_ld32(tbase + gi * 64, a);
            tmem_ld32(tbase + gi * 64 + 32, b2);
            tmem_ld_wait();
            const float inv = pack_y16(a, b2, pk);
            if (lane < wrows)
              p.yscale[static_cast<int64_t>(grow0 + lane) * (p.out_cols / 64) + col0 / 64] = inv;
            if (lane == 0) bulk_wait_read_all();  // the previous store has read the staging buffer
            __syncwarp();
#pragma unroll
            for (int v = 0; v < 8; ++v)
              *reinterpret_cast<uint4*>(stage + row_off + ((v ^ (lane & 7)) << 4)) =
                  make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          } else {
            uint32_t v32[32];
            if (!kIsFc2<MODE>) {
              uint32_t g[32];
              tmem_ld32(tbase + gi * 32, g);
              tmem_ld32(tbase + BN / 2 + gi * 32, v32);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                v32[i] = __float_as_uint(
                    round_tf32(silu_f(__uint_as_float(g[i])) * __uint_as_float(v32[i])));
            } else {
              tmem_ld32(tbase + gi * 32, v32);
              tmem_ld_wait();
            }
            if (lane == 0) bulk_wait_read_all();  // the previous store has read the staging buffer
            __syncwarp();
#pragma unroll
            for (int v = 0; v < 8; ++v)
              *reinterpret_cast<uint4*>(stage + row_off + ((v ^ (lane & 7)) << 4)) =
                  make_uint4(v32[4 * v], v32[4 * v + 1], v32[4 * v + 2], v32[4 * v + 3]);
          }
          if (wrows == 32) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOut, stage, col0, grow0);
              bulk_commit();
            }
            ++ngroups_tma;
          } else if (lane < wrows) {
            char* dst = static_cast<char*>(p.out) +
                        (static_cast<int64_t>(grow0 + lane) * p.out_cols + col0) *
                            (!kIsFc2<MODE> ? ES : 2);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<uint4*>(dst)[v] =
                  *reinterpret_cast<const uint4*>(stage + row_off + ((v ^ (lane & 7)) << 4));
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&tempty[acc]);
        else mbar_arrive_remote_relaxed(leader_tempty + acc * 8);  // after tcgen05.wait::ld
      }
      acc ^= 1;
      if (acc == 0) aph ^= 1;
      if constexpr (MODE == MODE_FC2C) {
        if (pend_wrows > 0) {
          bool pushed = true;
          if (lane == 0) {  // the previous tile's stores; this tile's may stay in flight
            bulk_wait_keep_n(ngroups_tma);
            fence_proxy_async_global();
            pushed = combine_push(cq + q, qs, qph, pend_n, pend_grow0, pend_wrows, ctl);
          }
          if (!__shfl_sync(0xffffffffu, pushed, 0)) break;
        }
        pend_grow0 = grow0;
        pend_wrows = wrows > 0 ? wrows : 0;
        pend_n = n;
      }
    }
    if (lane == 0) bulk_wait_all();
    if constexpr (MODE == MODE_FC2C) {
      if (lane == 0 && *abort_sh == 0) {
        fence_proxy_async_global();
        bool ok = true;
        if (pend_wrows > 0) ok = combine_push(cq + q, qs, qph, pend_n, pend_grow0, pend_wrows, ctl);
        if (ok) combine_push(cq + q, qs, qph, -1, 0, 0, ctl);  // no more work
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, P_TMEM_COLS);
}

// ----------------------------------------------------------------------------
// combine (unpermute with probs): out[t, :] = sum_j probs[t, j] * y(t, j) over
// valid pairs, y(t, j) the fc2 row unpermute_dst[t*k + j] decoded from fp16
// times its exact power-of-two factor; products rounded to fp32 and summed in
// ascending j, so the result is bitwise reproducible.
// ----------------------------------------------------------------------------
// One thread per 8 output columns of a token.  KC > 0: k == KC is known at
// compile time, so the k row indices, weights, factors and 16-byte row loads
// are all issued before the first add (k loads in flight per thread instead
// of one); KC == 0 is the same sum for any k, one slot at a time.
template <int KC>
__global__ void combine_kernel(const __half* __restrict__ y, const float* __restrict__ yscale,
                               const float* __restrict__ probs, const int32_t* __restrict__ offsets,
                               const int32_t* __restrict__ unpermute_dst, void* __restrict__ out,
                               int64_t T, int H, int k, int E, int out_bf16) {
  const int64_t H8 = H / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= T * H8) return;
  griddep_wait();
  griddep_launch_dependents();
  const int64_t t = idx / H8;
  const int c = static_cast<int>(idx - t * H8) * 8;
  const int32_t nvalid = __ldg(offsets + E);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  auto add = [&](float pj, float f, const uint4& raw) {
    const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = __half22float2(h2[i]);
      acc[2 * i] += __fmul_rn(pj, v.x * f);
      acc[2 * i + 1] += __fmul_rn(pj, v.y * f);
    }
  };
  if constexpr (KC > 0) {
    int32_t row[KC];
    float pj[KC], f[KC];
    uint4 raw[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      row[j] = __ldg(unpermute_dst + t * KC + j);
      pj[j] = __ldg(probs + t * KC + j);
    }
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      const bool ok = row[j] < nvalid;
      const int32_t r = ok ? row[j] : 0;
      f[j] = ok ? __ldg(yscale + static_cast<int64_t>(r) * (H / 64) + c / 64) : 0.f;
      raw[j] = ok ? __ldg(reinterpret_cast<const uint4*>(y + static_cast<int64_t>(r) * H + c))
                  : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < KC; ++j)
      if (row[j] < nvalid) add(pj[j], f[j], raw[j]);
  } else {
    for (int j = 0; j < k; ++j) {
      const int64_t flat = t * k + j;
      const int32_t r = __ldg(unpermute_dst + flat);
      if (r >= nvalid) continue;
      add(__ldg(probs + flat), __ldg(yscale + static_cast<int64_t>(r) * (H / 64) + c / 64),
          __ldg(reinterpret_cast<const uint4*>(y + static_cast<int64_t>(r) * H + c)));
    }
  }
  if (out_bf16) {
    uint4 w;
    w.x = pack_bf16x2(acc[0], acc[1]);
    w.y = pack_bf16x2(acc[2], acc[3]);
    w.z = pack_bf16x2(acc[4], acc[5]);
    w.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + t * H + c) = w;
  } else {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + t * H + c);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

__global__ void round_tf32_kernel(const float* __restrict__ src, float* __restrict__ dst, size_t n) {
  griddep_wait();
  griddep_launch_dependents();
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (; i < n; i += stride) dst[i] = round_tf32(src[i]);
}

// dst[b, c, r] = tf32_round(src[b, r, c]) for src [batch, rows, cols]
__global__ void transpose_round_tf32_kernel(const float* __restrict__ src, float* __restrict__ dst,
                                            int rows, int cols) {
  __shared__ float tile[32][33];
  const int64_t b = blockIdx.z;
  const float* s = src + b * rows * static_cast<int64_t>(cols);
  float* d = dst + b * rows * static_cast<int64_t>(cols);
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  griddep_wait();
  griddep_launch_dependents();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = s[static_cast<int64_t>(r) * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) d[static_cast<int64_t>(c) * rows + r] = round_tf32(tile[threadIdx.x][i]);
  }
}

__global__ void selftest_wait_kernel(uint64_t limit_ns, int32_t* dev_status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtl ctl{&abort_flag, limit_ns, dev_status};
    mbar_wait(&bar, 0, ctl);  // nothing ever arrives: runs out after limit_ns
  }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int MODE, int ES>
static cudaError_t launch_one(const GemmArgs& g, cudaStream_t st) {
  const mc2_shape_t& s = *g.s;
  using TR = ElemTraits<ES>;
  const CUtensorMapDataType dt =
      ES == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const int64_t R = static_cast<int64_t>(s.T) * s.k;
  CUtensorMap tA, tB, tOut;
  GemmParams p;
  p.a_ptr = g.a;
  p.yscale = g.yscale;
  p.offsets = g.offsets;
  p.permute_src = g.permute_src;
  p.out = g.out;
  p.dev_status = g.dev_status;
  p.E = s.E;
  p.k = s.k;
  p.I = s.I;
  p.wait_limit_ns = wait_limit_ns();
  p.probs = g.probs;
  p.unpermute_dst = g.unpermute_dst;
  p.ctr = g.ctr;
  p.defer_items = g.defer_items;
  p.defer_count = g.defer_count;
  p.comb_out = g.comb_out;
  p.out_f32 = g.out_dtype == MC2_F32 ? 1 : 0;
  bool ok;
  if (!kIsFc2<MODE>) {
    p.K = s.H;
    p.n_tiles = (s.I + BN / 2 - 1) / (BN / 2);
    p.out_cols = s.I;
    ok = (TR::B_KMAJOR ? encode_3d(&tB, dt, ES, g.b, s.H, 2ull * s.I, s.E, TR::BK, BN / 2)
                       : encode_b_blocked(&tB, g.b, s.H, 2ull * s.I, s.E, 2, TR::BK, NB1 / 2, 2)) &&
         encode_2d(&tOut, dt, ES, g.out, MODE == MODE_FC1_PRE ? 2ull * s.I : s.I, R, 128 / ES, 32);
    if (MODE == MODE_FC1_ROWS)  // already permuted rows [R, H]: plain TMA tiles
      ok = ok && encode_2d(&tA, dt, ES, g.a, s.H, R, 128 / ES, BM);
    else
      tA = tB;  // unused: fc1's A rows are gathered with cp.async
  } else {
    p.K = s.I;
    p.n_tiles = (s.H + BN - 1) / BN;
    p.out_cols = s.H;
    ok = encode_2d(&tA, dt, ES, g.a, s.I, R, 128 / ES, BM) &&
         (TR::B_KMAJOR ? encode_3d(&tB, dt, ES, g.b, s.I, s.H, s.E, TR::BK, BN)
                       : encode_b_blocked(&tB, g.b, s.I, s.H, s.E, 1, TR::BK, NB1, 1)) &&
         encode_2d(&tOut, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.out, s.H, R, 64, 32);
  }
  if (!ok) return cudaErrorInvalidValue;
  constexpr size_t fixed = SMEM_BYTES_FIXED + kQueueBytes<MODE>;
  const size_t smem = fixed + (s.E + 1) * sizeof(int32_t);
  static PerDevice<KernelSetup> setup;
  const KernelSetup su = once_per_device(setup, [] {
    return setup_kernel(gmm_kernel<MODE, ES>, fixed + 1025 * sizeof(int32_t),
                        Roles<MODE>::kThreads, false);
  });
  if (su.err != cudaSuccess) return su.err;
  const int64_t tiles_upper = (R / BM + s.E) * static_cast<int64_t>(p.n_tiles);
  const int grid = static_cast<int>(std::min<int64_t>(num_sms(), std::max<int64_t>(tiles_upper, 1)));
  return launch_kernel(gmm_kernel<MODE, ES>, dim3(grid), dim3(Roles<MODE>::kThreads), smem,
                       st, 1, tA, tB, tOut, p);
}

template <int MODE, int ES>
static cudaError_t launch_pair(const GemmArgs& g, cudaStream_t st) {
  const mc2_shape_t& s = *g.s;
  using TR = ElemTraits<ES>;
  const CUtensorMapDataType dt =
      ES == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const int64_t R = static_cast<int64_t>(s.T) * s.k;
  CUtensorMap tA, tB, tOut;
  GemmParams p;
  p.a_ptr = g.a;
  p.yscale = g.yscale;
  p.offsets = g.offsets;
  p.permute_src = g.permute_src;
  p.out = g.out;
  p.dev_status = g.dev_status;
  p.E = s.E;
  p.k = s.k;
  p.I = s.I;
  p.wait_limit_ns = wait_limit_ns();
  p.probs = g.probs;
  p.unpermute_dst = g.unpermute_dst;
  p.ctr = g.ctr;
  p.defer_items = g.defer_items;
  p.defer_count = g.defer_count;
  p.comb_out = g.comb_out;
  p.out_f32 = g.out_dtype == MC2_F32 ? 1 : 0;
  bool ok;
  if (!kIsFc2<MODE>) {
    p.K = s.H;
    p.n_tiles = (s.I + BN / 2 - 1) / (BN / 2);
    p.out_cols = s.I;
    ok = (TR::B_KMAJOR ? encode_3d(&tB, dt, ES, g.b, s.H, 2ull * s.I, s.E, TR::BK, BN / 2)
                       : encode_b_blocked(&tB, g.b, s.H, 2ull * s.I, s.E, 2, TR::BK, NB1 / 2, 1)) &&
         encode_2d(&tOut, dt, ES, g.out, s.I, R, 128 / ES, 32);
    if (MODE == MODE_FC1_ROWS)  // already permuted rows [R, H]: plain TMA tiles
      ok = ok && encode_2d(&tA, dt, ES, g.a, s.H, R, 128 / ES, BM);
    else
      tA = tB;  // unused: fc1's A rows are gathered with cp.async
  } else {
    p.K = s.I;
    p.n_tiles = (s.H + BN - 1) / BN;
    p.out_cols = s.H;
    ok = encode_2d(&tA, dt, ES, g.a, s.I, R, 128 / ES, BM) &&
         (TR::B_KMAJOR ? encode_3d(&tB, dt, ES, g.b, s.I, s.H, s.E, TR::BK, BN / 2)
                       : encode_b_blocked(&tB, g.b, s.I, s.H, s.E, 1, TR::BK, NB1 / 2, 1)) &&
         encode_2d(&tOut, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.out, s.H, R, 64, 32);
  }
  if (!ok) return cudaErrorInvalidValue;
  constexpr size_t fixed = P_SMEM_BYTES_FIXED + kQueueBytes<MODE>;
  const size_t smem = fixed + (s.E + 1) * sizeof(int32_t);
  static PerDevice<KernelSetup> setup;
  const KernelSetup su = once_per_device(setup, [] {
    return setup_kernel(gmm_pair_kernel<MODE, ES>, fixed + 1025 * sizeof(int32_t),
                        Roles<MODE>::kThreads, true);
  });
  if (su.err != cudaSuccess) return su.err;
  // Persistent grid: exactly as many pairs as can be resident at once.  A
  // pair needs two SMs of one GPC, so this can be fewer than SMs / 2; any
  // cluster beyond it would run its whole tile list as a second wave.
  const int max_clusters = su.pair_clusters;
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  const int64_t pair_tiles_upper = (R / (2 * BM) + s.E) * static_cast<int64_t>(p.n_tiles);
  const int grid = 2 * static_cast<int>(std::min<int64_t>(max_clusters,
                                                          std::max<int64_t>(pair_tiles_upper, 1)));
  return launch_kernel(gmm_pair_kernel<MODE, ES>, dim3(grid), dim3(Roles<MODE>::kThreads), smem,
                       st, 2, tA, tB, tOut, p);
}

// Automatic choice, from measurements on GB300 (4096- and 16384-token
// workloads): CTA pairs win for fc2 when experts average >= 256 rows (fc2 +
// combine 125 vs 135 us and 400 vs 430 us, although 256-row tiles pad a
// fifth of the 4096-token rows against a ninth for 128-row tiles) and lose
// for fc1 (206 vs 191 us, 617 vs 583 us); with few rows per expert
// (decode-like batches) single CTAs waste less tensor work on padding and are
// already bound by weight streaming.
static bool use_pairs(const mc2_shape_t& s, int mode) {
  const int forced = tile_pairing_override();
  if (forced == 1) return false;
  if (forced == 2) return num_sms() >= 2;
  const int64_t R = static_cast<int64_t>(s.T) * s.k;
  return (mode == MODE_FC2 || mode == MODE_FC2C) && num_sms() >= 2 &&
         R >= 2 * BM * static_cast<int64_t>(s.E);
}

bool fused_combine_supported(const mc2_shape_t& s) {
  const int64_t items = static_cast<int64_t>(s.T) * ((s.H + BN - 1) / BN);
  return s.k >= 1 && s.k <= KMAX_FUSED && items < (int64_t(1) << 31);
}

// Before a fused fc2 + combine: every (token, column tile) counter starts at
// k minus the token's valid slots (so the last of its rows brings it to k),
// and a token with no valid slot gets its zero output row here (no fc2 row
// will ever complete it).  One thread per token.
__global__ void combine_prep_kernel(const int32_t* __restrict__ offsets,
                                    const int32_t* __restrict__ unpermute_dst, int32_t* ctr,
                                    int32_t* defer_count, void* out, int64_t T, int k, int E,
                                    int H, int n_tiles, int out_f32) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t == 0) *defer_count = 0;
  if (t >= T) return;
  const int32_t nvalid = __ldg(offsets + E);
  int valid = 0;
  for (int j = 0; j < k; ++j) valid += __ldg(unpermute_dst + t * k + j) < nvalid;
  for (int n = 0; n < n_tiles; ++n) ctr[t * n_tiles + n] = k - valid;
  if (valid == 0) {
    if (out_f32) {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + t * H);
      for (int c = 0; c < H / 4; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + t * H);
      for (int c = 0; c < H / 8; ++c) o[c] = make_uint4(0, 0, 0, 0);
    }
  }
}

static cudaError_t launch_combine_prep(const GemmArgs& g, cudaStream_t st) {
  const mc2_shape_t& s = *g.s;
  const int threads = 256;
  const int64_t blocks = (static_cast<int64_t>(s.T) + threads - 1) / threads;
  const cudaError_t e = launch_kernel(
      combine_prep_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, st, 1,
      g.offsets, g.unpermute_dst, g.ctr, g.defer_count, g.comb_out, static_cast<int64_t>(s.T),
      static_cast<int>(s.k), static_cast<int>(s.E), static_cast<int>(s.H), (s.H + BN - 1) / BN,
      g.out_dtype == MC2_F32 ? 1 : 0);
  note_launches(1);
  return e;
}

// After a fused fc2 + combine: the (token, column tile) sums the combine
// warps deferred, one per warp iteration, over a grid-stride loop.
__global__ void __launch_bounds__(256) combine_deferred_kernel(
    const __half* __restrict__ y, const float* __restrict__ yscale,
    const float* __restrict__ probs, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ unpermute_dst, const int32_t* __restrict__ items,
    const int32_t* __restrict__ count, void* out, int H, int k, int E, int n_tiles,
    int out_f32) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int n_items = *count;
  CombineArgs a;
  a.y = y;
  a.yscale = yscale;
  a.out = out;
  a.H = H;
  a.out_f32 = out_f32;
  a.nvalid = __ldg(offsets + E);
  for (int64_t i = warp; i < n_items; i += nwarps) {
    const int item = __ldg(items + i);
    const int t[1] = {item / n_tiles};
    const int col[1] = {(item - t[0] * n_tiles) * BN + 8 * lane};
    int32_t r[1][KMAX_FUSED];
    float pj[1][KMAX_FUSED];
#pragma unroll
    for (int j = 0; j < KMAX_FUSED; ++j) {
      r[0][j] = j < k ? __ldg(unpermute_dst + static_cast<int64_t>(t[0]) * k + j) : a.nvalid;
      pj[0][j] = j < k ? __ldg(probs + static_cast<int64_t>(t[0]) * k + j) : 0.f;
    }
    combine_jobs<1>(a, t, col, r, pj);
  }
}

static cudaError_t launch_combine_deferred(const GemmArgs& g, cudaStream_t st) {
  const mc2_shape_t& s = *g.s;
  const cudaError_t e = launch_kernel(
      combine_deferred_kernel, dim3(static_cast<unsigned>(num_sms() * 8)), dim3(256), 0, st, 1,
      static_cast<const __half*>(g.out), g.yscale, g.probs, g.offsets, g.unpermute_dst,
      g.defer_items, g.defer_count, g.comb_out, static_cast<int>(s.H), static_cast<int>(s.k),
      static_cast<int>(s.E), (s.H + BN - 1) / BN, g.out_dtype == MC2_F32 ? 1 : 0);
  note_launches(1);
  return e;
}

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t st) {
  if (static_cast<int64_t>(g.s->T) * g.s->k == 0) return cudaSuccess;
  cudaError_t e;
  const bool pairs = use_pairs(*g.s, g.mode);
  if (g.mode == MODE_FC1) {
    if (pairs)
      e = g.a_elem_bytes == 2 ? launch_pair<MODE_FC1, 2>(g, st) : launch_pair<MODE_FC1, 4>(g, st);
    else
      e = g.a_elem_bytes == 2 ? launch_one<MODE_FC1, 2>(g, st) : launch_one<MODE_FC1, 4>(g, st);
  } else if (g.mode == MODE_FC1_PRE) {  // bf16, single CTAs
    if (g.a_elem_bytes != 2) return cudaErrorInvalidValue;
    e = launch_one<MODE_FC1_PRE, 2>(g, st);
  } else if (g.mode == MODE_FC1_ROWS) {  // bf16 only
    if (g.a_elem_bytes != 2) return cudaErrorInvalidValue;
    e = pairs ? launch_pair<MODE_FC1_ROWS, 2>(g, st) : launch_one<MODE_FC1_ROWS, 2>(g, st);
  } else if (g.mode == MODE_FC2C) {  // fc2 with the weighted combine fused in
    if (!fused_combine_supported(*g.s) || !g.probs || !g.unpermute_dst || !g.ctr ||
        !g.defer_items || !g.defer_count || !g.comb_out)
      return cudaErrorInvalidValue;
    e = launch_combine_prep(g, st);
    if (e != cudaSuccess) return e;
    if (pairs)
      e = g.a_elem_bytes == 2 ? launch_pair<MODE_FC2C, 2>(g, st) : launch_pair<MODE_FC2C, 4>(g, st);
    else
      e = g.a_elem_bytes == 2 ? launch_one<MODE_FC2C, 2>(g, st) : launch_one<MODE_FC2C, 4>(g, st);
    note_launches(1);
    if (e == cudaSuccess) e = launch_combine_deferred(g, st);
    return e;
  } else {
    if (pairs)
      e = g.a_elem_bytes == 2 ? launch_pair<MODE_FC2, 2>(g, st) : launch_pair<MODE_FC2, 4>(g, st);
    else
      e = g.a_elem_bytes == 2 ? launch_one<MODE_FC2, 2>(g, st) : launch_one<MODE_FC2, 4>(g, st);
  }
  note_launches(1);
  return e;
}

cudaError_t launch_combine(const mc2_shape_t& s, const void* y, const float* yscale,
                           const float* probs, const int32_t* offsets,
                           const int32_t* unpermute_dst, void* out, int out_dtype,
                           cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(s.T) * (s.H / 8);
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  decltype(&combine_kernel<0>) kern;
  switch (s.k) {
    case 1: kern = combine_kernel<1>; break;
    case 2: kern = combine_kernel<2>; break;
    case 4: kern = combine_kernel<4>; break;
    case 6: kern = combine_kernel<6>; break;
    case 8: kern = combine_kernel<8>; break;
    default: kern = combine_kernel<0>; break;
  }
  const cudaError_t e = launch_kernel(
      kern, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, st, 1,
      static_cast<const __half*>(y), yscale, probs, offsets, unpermute_dst, out,
      static_cast<int64_t>(s.T), static_cast<int>(s.H), static_cast<int>(s.k),
      static_cast<int>(s.E), out_dtype == MC2_BF16 ? 1 : 0);
  note_launches(1);
  return e;
}

// Materialised permute of the non-fused path: xp[p, :] = x[permute_src[p] / k, :]
// for every permuted row (16 bytes per thread).
// xp[p, :] = x[permute_src[p] / k, :]: one block per 8 permuted rows, each
// thread copying one 16-byte column of all 8 rows per step (8 row loads in
// flight per thread, one index load per row).
constexpr int PR_ROWS = 8;
constexpr int PR_THREADS = 128;

__global__ void permute_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ src,
                                    int k, int64_t R, int H8, uint4* __restrict__ xp) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * PR_ROWS;
  int64_t tok[PR_ROWS];
#pragma unroll
  for (int r = 0; r < PR_ROWS; ++r)
    tok[r] = row0 + r < R ? static_cast<int64_t>(__ldg(src + row0 + r) / k) : -1;
  for (int c = threadIdx.x; c < H8; c += PR_THREADS) {
    uint4 v[PR_ROWS];
#pragma unroll
    for (int r = 0; r < PR_ROWS; ++r)
      if (tok[r] >= 0) v[r] = __ldg(x + tok[r] * H8 + c);
#pragma unroll
    for (int r = 0; r < PR_ROWS; ++r)
      if (tok[r] >= 0) xp[(row0 + r) * H8 + c] = v[r];
  }
}

cudaError_t launch_permute_rows(const mc2_shape_t& s, const void* x, const int32_t* permute_src,
                                void* xp, cudaStream_t st) {
  const int64_t R = static_cast<int64_t>(s.T) * s.k;
  const int H8 = s.H / 8;  // bf16: 8 per 16 bytes
  if (R == 0) return cudaSuccess;
  const int64_t blocks = (R + PR_ROWS - 1) / PR_ROWS;
  const cudaError_t e = launch_kernel(permute_rows_kernel, dim3(static_cast<unsigned>(blocks)),
                                      dim3(PR_THREADS), 0, st, 1, static_cast<const uint4*>(x),
                                      permute_src, static_cast<int>(s.k), R, H8,
                                      static_cast<uint4*>(xp));
  note_launches(1);
  return e;
}

cudaError_t launch_round_tf32(const float* src, float* dst, size_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const size_t want = (n + threads - 1) / threads;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>(want, 152 * 16));
  const cudaError_t e = launch_kernel(round_tf32_kernel, dim3(blocks), dim3(threads), 0, st, 1,
                                      src, dst, n);
  note_launches(1);
  return e;
}

cudaError_t launch_transpose_round_tf32(const float* src, float* dst, int batch, int rows,
                                       int cols, cudaStream_t st) {
  if (static_cast<int64_t>(batch) * rows * cols == 0) return cudaSuccess;
  dim3 grid((cols + 31) / 32, (rows + 31) / 32, batch);
  const cudaError_t e = launch_kernel(transpose_round_tf32_kernel, grid, dim3(32, 8), 0, st, 1,
                                      src, dst, rows, cols);
  note_launches(1);
  return e;
}

cudaError_t launch_selftest_wait(uint64_t limit_ns, int32_t* dev_status, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(limit_ns, dev_status);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace mc2
