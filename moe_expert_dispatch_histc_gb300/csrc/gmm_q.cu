// gmm_q.cu -- the int8 path of the block: the dequantised grouped matmuls of
// "torch_npu.npu_mm_reduce_scatter_base" (Ascend op-plugin docs, "Function
// description"): out = (x1_scale * x2_scale) * (x1 @ x2), per-token x1_scale,
// per-channel x2_scale, no bias.
//
// sm_103a has no tcgen05 integer MMA (ptxas rejects .kind::i8 for it), so the
// int8 products run exactly on the bf16 tensor cores: every int8 value is a
// bf16 value, every product (|p| <= 127*127) is exact in the fp32
// accumulator, and every partial sum stays exact while |sum| < 2^24.  K is
// therefore cut into chunks of at most 1024 (1024 * 127^2 < 2^24), each chunk
// accumulates into its own TMEM region, and the epilogue converts the chunk
// sums to int32 and adds them: the result is the exact int32 product.
//
//   fc1: acc1 = x_q[tok] @ w1_q[e]; G = (xs[tok] * w1s[e, n]) * acc1;
//        h = silu(G_gate) * G_up (fp32) -> requant_rows -> h_q (int8), hs
//   fc2: acc2 = h_q @ w2_q[e];  y = (hs[p] * w2s[e, n]) * acc2 -> scaled fp16 -> combine
//
// Tiles are 128 x 128 (fc1: 64 gate + 64 up columns), 6 stages of 32 KB, one
// CTA per SM, the same warp roles as the bf16 kernel; or (when the tile
// pairing is forced) 256 x 128 tiles on CTA pairs (cta_group::2: each
// CTA streams its 128 rows and one 64-column block of B, 24 KB per stage, 8
// stages; fc2's odd CTA loads onto the even CTA's stage barrier, fc1's odd CTA
// relays its gathered stages).  TMEM is a ring of four
// 128-column chunk slots: chunk g of a CTA accumulates in slot g % 4, the
// epilogue reads a tile's chunks once its last one is committed and then frees
// their slots, so the MMAs of the next tile run during the epilogue (two tiles
// in flight for K <= 2048, one chunk ahead for K <= 3072).  Operands are bf16
// copies of the int8 tensors: weights expanded once by mc2_prepack_weights,
// x and h_q per call.
#include <algorithm>

#include "gmm_common.cuh"

namespace mc2 {

constexpr int QBN = 128;                       // UMMA N
constexpr int QCHUNK_KB = 16;                  // k-blocks (of 64) per exact fp32 chunk: K 1024
constexpr int QMAX_CHUNKS = 4;                 // K <= 4096
constexpr int QSLOTS = 4;                      // TMEM chunk slots of QBN columns (512 in all)

struct QParams {
  const void* a_ptr;           // fc1: x as bf16 [T, H] (gathered)
  const int32_t* offsets;
  const int32_t* permute_src;
  const float* a_scale;        // fc1: xs [T] (per token); fc2: hs [R] (per permuted row)
  const float* b_scale;        // fc1: w1s [E, 2I]; fc2: w2s [E, H]
  void* out;                   // raw: int32 acc; else fc1 h fp32 [R, I], fc2 y fp16 [R, H]
  float* yscale;               // fc2: decode factor per (row, 64 columns)
  int32_t* dev_status;
  int E, k, K, n_tiles, I, H, nchunk, raw;
  uint64_t wait_limit_ns;
};

template <int MODE>
struct QRoles {
  static constexpr int kGatherWarps = MODE == MODE_FC1 ? 4 : 0;
  static constexpr int kThreads = (6 + kGatherWarps) * 32;
};

// Pipeline geometry.  Single CTA: 128 x 128 tiles, a 16 KB B stage (two 64-
// column blocks).  CTA pair (cta_group::2, UMMA M = 256, N = 128): each CTA
// holds 128 rows of A and one 64-column block of B (fc1: the even CTA the gate
// block, the odd CTA the matching up block; fc2: the first or second 64 of the
// 128 output columns), 24 KB per stage instead of 32 KB, eight stages; each
// CTA's TMEM holds its 128 rows x all 128 columns, so the epilogue is the
// single-CTA one.
template <bool PAIR>
struct QGeom {
  static constexpr int kStages = PAIR ? 8 : 6;
  static constexpr int kBStage = PAIR ? 8192 : 16384;
  static constexpr int kStageBytes = A_STAGE + kBStage;
  static constexpr size_t kSmemFixed = 1024 + static_cast<size_t>(kStages) * kStageBytes +
                                       4 * OUT_STAGE + 512;
};

template <int MODE, bool PAIR>
__global__ void __launch_bounds__(QRoles<MODE>::kThreads, 1)
    gmm_q_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmOut, const QParams p) {
  using G = QGeom<PAIR>;
  constexpr int BK = 64;
  constexpr int STAGES = G::kStages;
  constexpr int B_STAGE = G::kBStage;
  constexpr int B_BLOCK = BK * 128;          // 64 K rows x 64 columns
  constexpr int KK_B = 16 * 128;             // B bytes per UMMA K step
  constexpr int TM = PAIR ? 2 * BM : BM;     // rows per tile
  constexpr uint32_t IDESC = instr_desc(1, false, true, TM, QBN);
  constexpr bool GATHER = MODE == MODE_FC1;
  // pair with TMA-loaded A: the odd CTA's copies complete on the even CTA's
  // full[s]; pair with gathered rows: the odd CTA relays its stages (pfull)
  constexpr bool DIRECT = PAIR && !GATHER;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE;
  uint8_t* sOut = sB + STAGES * B_STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + 4 * OUT_STAGE);
  uint64_t* pfull = full + STAGES;
  uint64_t* empty = pfull + STAGES;
  uint64_t* tfull = empty + STAGES;         // per TMEM chunk slot
  uint64_t* tempty = tfull + QSLOTS;
  uint64_t* mma_done = tempty + QSLOTS;
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_sh = reinterpret_cast<volatile int*>(tmem_base_sh + 1);
  int32_t* prefix = reinterpret_cast<int32_t*>(tmem_base_sh + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int nchunk = p.nchunk;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int nunits = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], GATHER ? 1 + 32 * QRoles<MODE>::kGatherWarps : 1);
      mbar_init(&pfull[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < QSLOTS; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], PAIR ? 2 * 4 : 4);  // one arrival per epilogue warp (of both CTAs)
    }
    mbar_init(mma_done, 1);
    *abort_sh = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    if (!GATHER) tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (!p.raw) tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_base_sh, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_base_sh, TMEM_COLS);
      tmem_relinquish();
    }
  }
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 2) {  // per-expert tile prefix: ceil(rows_e / TM) * n_tiles
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int t = 0;
      if (e < E) {
        const int rows = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
        t = ((rows + TM - 1) / TM) * p.n_tiles;
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
  if constexpr (PAIR) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_sh;
  int total = prefix[E];
  if constexpr (PAIR) {  // the pair's MMAs write one TMEM address in both CTAs
    const uint32_t peer_base = ld_shared_cluster_u32(map_to_rank(tmem_base_sh, rank ^ 1u));
    if (peer_base != tmem_base) {
      if (threadIdx.x == 0 && p.dev_status) atomicOr(p.dev_status, 0x4);
      total = 0;
    }
  }
  WaitCtl ctl{abort_sh, p.wait_limit_ns, p.dev_status};
  const int kblocks = p.K / BK;

  // This CTA's rows of a tile: [row0, row0 + rows) (rows may be <= 0 for the
  // odd CTA of a pair tile at an expert's end); pair0 is the tile's first row.
  auto tile_rows = [&](int tile, int& e, int& n, int& pair0, int& row0, int& rows) {
    int r0, rr;
    decode_tile(tile, prefix, E, p.n_tiles, p.offsets, e, n, r0, rr);
    if constexpr (PAIR) {  // decode_tile counts in BM rows; a pair tile spans 2 * BM
      const int local = tile - prefix[e];
      const int m_pairs = (prefix[e + 1] - prefix[e]) / p.n_tiles;
      const int mp = local - (local / m_pairs) * m_pairs;
      pair0 = __ldg(p.offsets + e) + mp * TM;
      row0 = pair0 + static_cast<int>(rank) * BM;
      rows = __ldg(p.offsets + e + 1) - row0;
    } else {
      pair0 = r0;
      row0 = r0;
      rows = rr;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint32_t leader_full = PAIR ? map_to_rank(full, 0) : 0u;
    int s = 0;
    uint32_t ph = 0;
    int n_arm = 0;
    bool ok = true;
    for (int tile = unit; tile < total && ok; tile += nunits) {
      int e, n, pair0, row0, rows;
      tile_rows(tile, e, n, pair0, row0, rows);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (lane == 0) ok = PAIR ? mbar_wait_cluster(&empty[s], ph ^ 1, ctl)
                                 : mbar_wait(&empty[s], ph ^ 1, ctl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          uint8_t* a_dst = sA + s * A_STAGE;
          uint8_t* b_dst = sB + s * B_STAGE;
          const int k0 = kb * BK;
          // B through a blocked map (64-column blocks of 128 bytes): one box
          // per stage.  Single CTA: fc1 the gate block n and the up block n
          // ([half][k row][128 B]), fc2 blocks 2n and 2n + 1.  Pair: this
          // CTA's one block -- fc1 gate (even CTA) or up (odd CTA) block n,
          // fc2 block 2n + rank.
          if constexpr (PAIR) {
            if (DIRECT && !leader) {
              const uint32_t bar = leader_full + s * 8;
              tma_load_2d_pair(a_dst, &tmA, bar, k0, row0);
              if (MODE == MODE_FC1)
                tma_load_5d_pair(b_dst, &tmB, bar, 0, k0, n, static_cast<int>(rank), e);
              else
                tma_load_4d_pair(b_dst, &tmB, bar, 0, k0, 2 * n + static_cast<int>(rank), e);
            } else {
              mbar_arrive_expect_tx(&full[s], GATHER ? B_STAGE : 2 * G::kStageBytes);
              if (!GATHER) tma_load_2d(a_dst, &tmA, &full[s], k0, row0);
              if (MODE == MODE_FC1)
                tma_load_5d(b_dst, &tmB, &full[s], 0, k0, n, static_cast<int>(rank), e);
              else
                tma_load_4d(b_dst, &tmB, &full[s], 0, k0, 2 * n + static_cast<int>(rank), e);
            }
          } else {
            mbar_arrive_expect_tx(&full[s], GATHER ? B_STAGE : G::kStageBytes);
            if (!GATHER) tma_load_2d(a_dst, &tmA, &full[s], k0, row0);
            if (MODE == MODE_FC1)
              tma_load_5d(b_dst, &tmB, &full[s], 0, k0, n, 0, e);
            else
              tma_load_4d(b_dst, &tmB, &full[s], 0, k0, 2 * n, e);
          }
        }
        __syncwarp();
        ++n_arm;
        if (++s == STAGES) { s = 0; ph ^= 1; }
      }
    }
    if (lane == 0) {  // every armed stage has landed and every commit to it has arrived
      volatile int never = 0;
      WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
      for (int st = 0; st < STAGES && st < n_arm; ++st) {
        const int last = st + STAGES * ((n_arm - 1 - st) / STAGES);
        if (!DIRECT || leader) mbar_wait_cluster(&full[st], (last / STAGES) & 1, drain);
        if (PAIR) mbar_wait_cluster(&empty[st], (last / STAGES) & 1, drain);
      }
    }
  } else if (warp == 1) {
    if (leader) {
      // ---------------------------------------------------------- MMA issuer
      // Chunk g of this CTA (tiles in order, chunks within a tile) accumulates
      // in TMEM slot g % 4; a slot is reused once the epilogue has read it.
      int s = 0;
      uint32_t ph = 0;
      int g = 0;
      bool ok = true;
      for (int tile = unit; tile < total && ok; tile += nunits) {
        uint32_t d = 0;
        int slot = 0;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (kb % QCHUNK_KB == 0) {  // next chunk: wait until its slot is free
            slot = g & (QSLOTS - 1);
            if (lane == 0) {
              const uint32_t par = ((g / QSLOTS) & 1) ^ 1;
              ok = PAIR ? mbar_wait_cluster(&tempty[slot], par, ctl)
                        : mbar_wait(&tempty[slot], par, ctl);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            d = tmem_base + static_cast<uint32_t>(slot * QBN);
            ++g;
          }
          if (lane == 0) {
            ok = mbar_wait_cluster(&full[s], ph, ctl);
            if (ok && PAIR && !DIRECT) ok = mbar_wait_cluster(&pfull[s], ph, ctl);
            if (GATHER && ok) fence_proxy_async_smem();  // gathered rows -> async proxy
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a_base = smem_u32(sA + s * A_STAGE);
            const uint32_t b_base = smem_u32(sB + s * B_STAGE);
            const bool first_of_chunk = (kb % QCHUNK_KB) == 0;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
              const uint64_t bdesc = smem_desc_sw128(b_base + kk * KK_B, B_BLOCK, 1024);
              const uint32_t acc = (first_of_chunk && kk == 0) ? 0u : 1u;
              if constexpr (PAIR) umma_pair<0>(d, adesc, bdesc, IDESC, acc);
              else umma<0>(d, adesc, bdesc, IDESC, acc);
            }
            if constexpr (PAIR) umma_commit_pair(&empty[s], 0x3);
            else umma_commit(&empty[s]);
          }
          __syncwarp();
          if (++s == STAGES) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        if (lane == 0) {  // the tile's last chunk slot
          if constexpr (PAIR) umma_commit_pair(&tfull[slot], 0x3);
          else umma_commit(&tfull[slot]);
        }
        __syncwarp();
      }
      if (lane == 0) {
        if constexpr (PAIR) umma_commit_pair(mma_done, 0x1);
        else umma_commit(mma_done);
        volatile int never = 0;
        WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
        mbar_wait_cluster(mma_done, 0, drain);
      }
      __syncwarp();
    } else if (!DIRECT) {
      // ---------------------------------------------------------- relay (odd CTA of a pair)
      const uint32_t leader_pfull = map_to_rank(pfull, 0);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = unit; tile < total && ok; tile += nunits) {
        for (int kb = 0; kb < kblocks; ++kb) {
          if (lane == 0) {
            ok = mbar_wait(&full[s], ph, ctl);
            if (GATHER && ok) fence_proxy_async_smem();  // gathered rows -> async proxy
            if (ok) mbar_arrive_remote_relaxed(leader_pfull + s * 8);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (++s == STAGES) { s = 0; ph ^= 1; }
        }
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ fc1 row gather
    const int t = threadIdx.x - 6 * 32;
    const int chunk = t & 7, rsub = t >> 3;
    const char* xg = static_cast<const char*>(p.a_ptr);
    const int64_t row_bytes = static_cast<int64_t>(p.K) * 2;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tile = unit; tile < total && ok; tile += nunits) {
      int e, n, pair0, row0, rows;
      tile_rows(tile, e, n, pair0, row0, rows);
      const int tok0 = __ldg(p.permute_src + pair0) / p.k;  // a valid row for padding
      const char* src[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = rsub + 16 * i;
        const int tok = r < rows ? __ldg(p.permute_src + row0 + r) / p.k : tok0;
        src[i] = xg + tok * row_bytes + chunk * 16;
      }
      for (int kb = 0; kb < kblocks; ++kb) {
        if (lane == 0) ok = PAIR ? mbar_wait_cluster(&empty[s], ph ^ 1, ctl)
                                 : mbar_wait(&empty[s], ph ^ 1, ctl);
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
    const int q = warp & 3;
    uint8_t* stage = sOut + q * OUT_STAGE;
    const uint32_t row_off = static_cast<uint32_t>(lane) * 128;
    const uint32_t leader_tempty = PAIR ? map_to_rank(tempty, 0) : 0u;
    int g = 0;              // first chunk of the current tile (same count as the MMA warp)
    uint32_t tf_phase = 0;  // bit b: parity of the next tfull[b] completion
    for (int tile = unit; tile < total; tile += nunits) {
      int e, n, pair0, row0, rows;
      tile_rows(tile, e, n, pair0, row0, rows);
      bool ok = true;
      const int last = (g + nchunk - 1) & (QSLOTS - 1);
      if (lane == 0) {
        ok = PAIR ? mbar_wait_cluster(&tfull[last], (tf_phase >> last) & 1, ctl)
                  : mbar_wait(&tfull[last], (tf_phase >> last) & 1, ctl);
      }
      tf_phase ^= 1u << last;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int wrows = min(32, rows - q * 32);
      const int grow0 = row0 + q * 32;
      const int grow = grow0 + lane;
      const bool valid = lane < wrows;
      if (wrows > 0) {
        // per-row scale: fc1 the token's x scale, fc2 the row's h scale (the
        // raw test mode has no scales: the pointers may be null there)
        float rs = 0.f;
        if (valid && !p.raw)
          rs = MODE == MODE_FC1 ? __ldg(p.a_scale + __ldg(p.permute_src + grow) / p.k)
                                : __ldg(p.a_scale + grow);
        const float* cs = p.b_scale + static_cast<int64_t>(e) *
                                          (MODE == MODE_FC1 ? 2 * p.I : p.H);
        // fc1: two groups of 32 gate columns (+ the matching 32 up columns);
        // fc2: two groups of 64 columns (s0: the first 32, s1: the next 32)
        constexpr int NGROUPS = 2;
        constexpr int S1_OFF = MODE == MODE_FC1 ? 64 : 32;   // TMEM column offset of s1
        constexpr int GW = MODE == MODE_FC1 ? 32 : 64;       // group width in columns
#pragma unroll 1
        for (int gi = 0; gi < NGROUPS; ++gi) {
          const int col0 = n * (MODE == MODE_FC1 ? 64 : QBN) + gi * GW;
          if (MODE == MODE_FC2 && col0 >= p.H) break;
          // exact int32 sums over the K chunks of this group's columns
          int32_t s0[32], s1[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) { s0[i] = 0; s1[i] = 0; }
#pragma unroll 1
          for (int c = 0; c < nchunk; ++c) {
            const uint32_t cs_base = tbase + ((g + c) & (QSLOTS - 1)) * QBN;
            uint32_t v[32];
            tmem_ld32(cs_base + gi * GW, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) s0[i] += __float2int_rn(__uint_as_float(v[i]));
            tmem_ld32(cs_base + gi * GW + S1_OFF, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) s1[i] += __float2int_rn(__uint_as_float(v[i]));
          }
          if (p.raw) {  // test mode: the int32 accumulators themselves
            if (valid) {
              int32_t* o = static_cast<int32_t*>(p.out);
              int4* d0;
              int4* d1;
              if (MODE == MODE_FC1) {
                d0 = reinterpret_cast<int4*>(o + static_cast<int64_t>(grow) * 2 * p.I + col0);
                d1 = reinterpret_cast<int4*>(o + static_cast<int64_t>(grow) * 2 * p.I + p.I + col0);
              } else {
                d0 = reinterpret_cast<int4*>(o + static_cast<int64_t>(grow) * p.H + col0);
                d1 = reinterpret_cast<int4*>(o + static_cast<int64_t>(grow) * p.H + col0 + 32);
              }
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                d0[v] = make_int4(s0[4 * v], s0[4 * v + 1], s0[4 * v + 2], s0[4 * v + 3]);
                d1[v] = make_int4(s1[4 * v], s1[4 * v + 1], s1[4 * v + 2], s1[4 * v + 3]);
              }
            }
            continue;
          }
          // dequant: (row scale * column scale) * acc, in fp32
          uint32_t pk[32];
          if (MODE == MODE_FC1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float g = (rs * __ldg(cs + col0 + i)) * static_cast<float>(s0[i]);
              const float u = (rs * __ldg(cs + p.I + col0 + i)) * static_cast<float>(s1[i]);
              pk[i] = __float_as_uint(silu_f(g) * u);
            }
          } else {  // y as fp16 with a power-of-two scale per 64 columns
            uint32_t y0[32], y1[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              y0[i] = __float_as_uint((rs * __ldg(cs + col0 + i)) * static_cast<float>(s0[i]));
              y1[i] = __float_as_uint((rs * __ldg(cs + col0 + 32 + i)) * static_cast<float>(s1[i]));
            }
            const float inv = pack_y16(y0, y1, pk);
            if (valid) p.yscale[static_cast<int64_t>(grow) * (p.H / 64) + col0 / 64] = inv;
          }
          const int out_cols = MODE == MODE_FC1 ? p.I : p.H;
          constexpr int ESZ = MODE == MODE_FC1 ? 4 : 2;   // h fp32, y fp16
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<uint4*>(stage + row_off + ((v ^ (lane & 7)) << 4)) =
                make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          if (wrows == 32) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOut, stage, col0, grow0);
              bulk_commit();
            }
          } else if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(p.out) +
                                                  (static_cast<int64_t>(grow) * out_cols + col0) * ESZ);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = *reinterpret_cast<const uint4*>(stage + row_off + ((v ^ (lane & 7)) << 4));
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // free the tile's chunk slots (after tcgen05.wait::ld)
        for (int c = 0; c < nchunk; ++c) {
          const int sl = (g + c) & (QSLOTS - 1);
          if (!PAIR || leader) mbar_arrive(&tempty[sl]);
          else mbar_arrive_remote_relaxed(leader_tempty + sl * 8);
        }
      }
      g += nchunk;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  if constexpr (PAIR) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ----------------------------------------------------------------------------
// Wide int8 GEMM (the default single-CTA form): 128 x 256 tiles (fc1: 128
// gate + 128 up columns), four 48 KB stages -- the bf16 block's 48 KB of
// operands per 512 MMA cycles, where the 128 x 128 tiles above move 32 KB per
// 256 cycles.  TMEM holds two 256-column accumulator slots.  Tile t of a CTA
// has a first slot F = t mod 2 and a second slot S: chunk 0 of K (k < 1024)
// accumulates in F, every later chunk in S, and the epilogue folds each of
// them into F (tcgen05.ld, add, tcgen05.st), releasing S at once.  The next
// tile's chunk 0 therefore accumulates in S while the epilogue dequantises and
// stores the current tile from F.  The folds keep the running sum as exact
// fp32 integers while they stay below 2^24 and as int32 beyond; the last fold
// rounds once to fp32, the value the 128 x 128 kernel's dequant takes from
// its int32 sums, so both give the same bits.
// ----------------------------------------------------------------------------
constexpr int QW_BN = 256;
constexpr int QW_STAGES = 4;
constexpr int QW_B_STAGE = 32768;          // 64 K rows x 256 columns x 2 B
constexpr int QW_STAGE_BYTES = A_STAGE + QW_B_STAGE;
constexpr size_t QW_SMEM_FIXED = 1024 + static_cast<size_t>(QW_STAGES) * QW_STAGE_BYTES +
                                 4 * OUT_STAGE + 256;

__device__ __forceinline__ int32_t f2i(uint32_t v) { return __float2int_rn(__uint_as_float(v)); }

template <int MODE>
__global__ void __launch_bounds__(QRoles<MODE>::kThreads, 1)
    gmm_qw_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmOut, const QParams p) {
  constexpr int BK = 64;
  constexpr int STAGES = QW_STAGES;
  constexpr int B_STAGE = QW_B_STAGE;
  constexpr int B_BLOCK = BK * 128;          // 64 K rows x 64 columns
  constexpr int KK_B = 16 * 128;             // B bytes per UMMA K step
  constexpr uint32_t IDESC = instr_desc(1, false, true, BM, QW_BN);
  constexpr bool GATHER = MODE == MODE_FC1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE;
  uint8_t* sOut = sB + STAGES * B_STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + 4 * OUT_STAGE);
  uint64_t* empty = full + STAGES;
  uint64_t* done = empty + STAGES;     // [2]: a chunk is complete in the slot (MMA -> epilogue)
  uint64_t* sfree = done + 2;          // [2]: the slot has been read (epilogue -> MMA)
  uint64_t* mma_done = sfree + 2;
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_sh = reinterpret_cast<volatile int*>(tmem_base_sh + 1);
  int32_t* prefix = reinterpret_cast<int32_t*>(tmem_base_sh + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int nchunk = p.nchunk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], GATHER ? 1 + 32 * QRoles<MODE>::kGatherWarps : 1);
      mbar_init(&empty[s], 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&done[j], 1);
      mbar_init(&sfree[j], 4);  // lane 0 of each epilogue warp
    }
    mbar_init(mma_done, 1);
    *abort_sh = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    if (!GATHER) tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (!p.raw) tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_sh, TMEM_COLS);
    tmem_relinquish();
  }
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
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int e, n, row0, rows;
      decode_tile(tile, prefix, E, p.n_tiles, p.offsets, e, n, row0, rows);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1, ctl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          const int k0 = kb * BK;
          uint8_t* b_dst = sB + s * B_STAGE;
          mbar_arrive_expect_tx(&full[s], GATHER ? B_STAGE : QW_STAGE_BYTES);
          if (!GATHER) tma_load_2d(sA + s * A_STAGE, &tmA, &full[s], k0, row0);
          // B in one blocked box: fc1 gate blocks 2n, 2n+1 then the same up
          // blocks ([half][block][k row][128 B]); fc2 blocks 4n .. 4n+3
          if (MODE == MODE_FC1) tma_load_5d(b_dst, &tmB, &full[s], 0, k0, 2 * n, 0, e);
          else tma_load_4d(b_dst, &tmB, &full[s], 0, k0, 4 * n, e);
        }
        __syncwarp();
        ++n_arm;
        if (++s == STAGES) { s = 0; ph ^= 1; }
      }
    }
    if (lane == 0) {  // every armed stage has landed before the CTA can exit (bounded)
      volatile int never = 0;
      WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
      for (int st = 0; st < STAGES && st < n_arm; ++st) {
        const int last = st + STAGES * ((n_arm - 1 - st) / STAGES);
        mbar_wait(&full[st], (last / STAGES) & 1, drain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Each chunk starts a fresh accumulation in its slot once the epilogue
    // has released the slot's previous contents (the first use of each slot
    // passes at once: parity of the phase before the first).
    int s = 0;
    uint32_t ph = 0;
    uint32_t nwait = 0;  // bit j: parity of the waits on slot j so far
    bool ok = true;
    int lt = 0;  // tiles of this CTA so far
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++lt) {
      const int F = lt & 1;
      uint32_t d = 0;
      for (int kb = 0; kb < kblocks; ++kb) {
        const int c = kb / QCHUNK_KB;
        const bool first = (kb % QCHUNK_KB) == 0;
        const int slot = c == 0 ? F : F ^ 1;
        if (first) {
          if (lane == 0) ok = mbar_wait(&sfree[slot], ((nwait >> slot) & 1u) ^ 1u, ctl);
          nwait ^= 1u << slot;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          tc_fence_after();
          d = tmem_base + static_cast<uint32_t>(slot * QW_BN);
        }
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
            const uint64_t bdesc = smem_desc_sw128(b_base + kk * KK_B, B_BLOCK, 1024);
            umma<0>(d, adesc, bdesc, IDESC, (first && kk == 0) ? 0u : 1u);
          }
          umma_commit(&empty[s]);
          if ((kb % QCHUNK_KB) == QCHUNK_KB - 1 || kb == kblocks - 1)
            umma_commit(&done[slot]);  // the chunk is complete
        }
        __syncwarp();
        if (++s == STAGES) { s = 0; ph ^= 1; }
      }
    }
    if (lane == 0) {
      umma_commit(mma_done);
      volatile int never = 0;
      WaitCtl drain{&never, p.wait_limit_ns, p.dev_status};
      mbar_wait(mma_done, 0, drain);
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ------------------------------------------------------------ fc1 row gather
    const int t = threadIdx.x - 6 * 32;
    const int chunk = t & 7, rsub = t >> 3;
    const char* xg = static_cast<const char*>(p.a_ptr);
    const int64_t row_bytes = static_cast<int64_t>(p.K) * 2;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int e, n, row0, rows;
      decode_tile(tile, prefix, E, p.n_tiles, p.offsets, e, n, row0, rows);
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
    const int q = warp & 3;
    uint8_t* stage = sOut + q * OUT_STAGE;
    const uint32_t row_off = static_cast<uint32_t>(lane) * 128;
    uint32_t pd = 0;  // bit j: parity of the next completion of done[j]
    int lt = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++lt) {
      int e, n, row0, rows;
      decode_tile(tile, prefix, E, p.n_tiles, p.offsets, e, n, row0, rows);
      const int F = lt & 1, S = F ^ 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&done[F], (pd >> F) & 1u, ctl);
      pd ^= 1u << F;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tF = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(F * QW_BN);
      const uint32_t tS = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(S * QW_BN);
      const int wrows = min(32, rows - q * 32);
      const int grow0 = row0 + q * 32;
      const int grow = grow0 + lane;
      const bool valid = lane < wrows;
      // Representation of slot F per 64-column group (bit g of gint, the same
      // for the whole warp): fp32 or int32.  Every chunk sum is an exact fp32
      // integer below 2^24.  The dequant needs only fp32(sum), the
      // round-to-nearest value of the exact int32 sum.  A fold adds in fp32
      // while that stays exact (every |sum| of the warp's group below 2^24,
      // checked by a warp vote) and always at the last fold (one rounding of
      // the exact sum, which is fp32(sum)); otherwise the group switches to
      // exact int32.  The raw int32 output folds in int32 throughout.
      uint32_t gint = 0;
      for (int c = 1; c < nchunk; ++c) {  // fold each later chunk into F, then release S
        if (lane == 0) ok = mbar_wait(&done[S], (pd >> S) & 1u, ctl);
        pd ^= 1u << S;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        if (wrows > 0) {  // 64 columns per round trip: four loads behind one wait
#pragma unroll 1
          for (int g = 0; g < QW_BN / 64; ++g) {
            uint32_t va[2][32], vb[2][32];
            tmem_ld32(tF + g * 64, va[0]);
            tmem_ld32(tF + g * 64 + 32, va[1]);
            tmem_ld32(tS + g * 64, vb[0]);
            tmem_ld32(tS + g * 64 + 32, vb[1]);
            tmem_ld_wait();
            bool to_int = p.raw || ((gint >> g) & 1u);
            if (!to_int && c == nchunk - 1) {  // last fold: one rounding of the exact sum
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  va[h][i] = __float_as_uint(__uint_as_float(va[h][i]) + __uint_as_float(vb[h][i]));
            } else if (!to_int) {
              bool exact = true;
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  const float x = __uint_as_float(va[h][i]) + __uint_as_float(vb[h][i]);
                  exact = exact && fabsf(x) < 16777216.0f;
                  va[h][i] = __float_as_uint(x);
                }
              if (!__all_sync(0xffffffffu, exact)) {
                // rare: F's group is still unchanged in TMEM; fold it in int32
                tmem_ld32(tF + g * 64, va[0]);
                tmem_ld32(tF + g * 64 + 32, va[1]);
                tmem_ld_wait();
                to_int = true;
              }
            }
            if (to_int) {
              const bool fi = (gint >> g) & 1u;
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  va[h][i] = static_cast<uint32_t>(
                      (fi ? static_cast<int32_t>(va[h][i]) : f2i(va[h][i])) + f2i(vb[h][i]));
              gint |= 1u << g;
            }
            tmem_st32(tF + g * 64, va[0]);
            tmem_st32(tF + g * 64 + 32, va[1]);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfree[S]);
      }
      if (!ok) break;
      // exact int32 sums of the 32 columns at TMEM columns c0 and c1 of slot F
      // (two loads behind one wait)
      auto sums2x32 = [&](int c0, int c1, int32_t (&o0)[32], int32_t (&o1)[32]) {
        uint32_t va[32], vb[32];
        tmem_ld32(tF + c0, va);
        tmem_ld32(tF + c1, vb);
        tmem_ld_wait();
        const bool i0 = (gint >> (c0 >> 6)) & 1u, i1 = (gint >> (c1 >> 6)) & 1u;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          o0[i] = i0 ? static_cast<int32_t>(va[i]) : f2i(va[i]);
          o1[i] = i1 ? static_cast<int32_t>(vb[i]) : f2i(vb[i]);
        }
      };
      // the same sums rounded to fp32 (what the dequant multiplies): int32
      // slots are converted, fp32 slots already hold that value (a zero sum is
      // +0, as the conversion of int 0 gives)
      auto acc2x32 = [&](int c0, int c1, float (&o0)[32], float (&o1)[32]) {
        uint32_t va[32], vb[32];
        tmem_ld32(tF + c0, va);
        tmem_ld32(tF + c1, vb);
        tmem_ld_wait();
        const bool i0 = (gint >> (c0 >> 6)) & 1u, i1 = (gint >> (c1 >> 6)) & 1u;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float x0 = __uint_as_float(va[i]), x1 = __uint_as_float(vb[i]);
          o0[i] = i0 ? static_cast<float>(static_cast<int32_t>(va[i])) : (x0 == 0.f ? 0.f : x0);
          o1[i] = i1 ? static_cast<float>(static_cast<int32_t>(vb[i])) : (x1 == 0.f ? 0.f : x1);
        }
      };
      if (wrows > 0) {
        float rs = 0.f;
        if (valid && !p.raw)
          rs = MODE == MODE_FC1 ? __ldg(p.a_scale + __ldg(p.permute_src + grow) / p.k)
                                : __ldg(p.a_scale + grow);
        const float* cs = p.b_scale + static_cast<int64_t>(e) *
                                          (MODE == MODE_FC1 ? 2 * p.I : p.H);
        // fc1: four groups of 32 gate columns (+ the matching up columns);
        // fc2: four groups of 64 columns (s0: the first 32, s1: the next 32)
        constexpr int GW = MODE == MODE_FC1 ? 32 : 64;
#pragma unroll 1
        for (int gi = 0; gi < 4; ++gi) {
          const int col0 = n * (MODE == MODE_FC1 ? 128 : QW_BN) + gi * GW;
          if (col0 >= (MODE == MODE_FC1 ? p.I : p.H)) break;
          if (p.raw) {  // test mode: the int32 accumulators themselves
            int32_t s0[32], s1[32];
            if (MODE == MODE_FC1) sums2x32(gi * 32, 128 + gi * 32, s0, s1);  // gate, up
            else sums2x32(gi * 64, gi * 64 + 32, s0, s1);
            if (valid) {
              int32_t* o = static_cast<int32_t*>(p.out);
              int4* d0;
              int4* d1;
              if (MODE == MODE_FC1) {
                d0 = reinterpret_cast<int4*>(o + static_cast<int64_t>(grow) * 2 * p.I + col0);
                d1 = reinterpret_cast<int4*>(o + static_cast<int64_t>(grow) * 2 * p.I + p.I + col0);
              } else {
                d0 = reinterpret_cast<int4*>(o + static_cast<int64_t>(grow) * p.H + col0);
                d1 = reinterpret_cast<int4*>(o + static_cast<int64_t>(grow) * p.H + col0 + 32);
              }
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                d0[v] = make_int4(s0[4 * v], s0[4 * v + 1], s0[4 * v + 2], s0[4 * v + 3]);
                d1[v] = make_int4(s1[4 * v], s1[4 * v + 1], s1[4 * v + 2], s1[4 * v + 3]);
              }
            }
            continue;
          }
          // dequant: (row scale * column scale) * acc, in fp32
          float s0[32], s1[32];
          if (MODE == MODE_FC1) acc2x32(gi * 32, 128 + gi * 32, s0, s1);  // gate, up
          else acc2x32(gi * 64, gi * 64 + 32, s0, s1);
          uint32_t pk[32];
          // column scales as float4 loads (16-byte aligned: the scale rows
          // start at multiples of 64 columns and col0 is a multiple of 32)
          const float4* c0 = reinterpret_cast<const float4*>(cs + col0);
          const float4* c1 = reinterpret_cast<const float4*>(
              cs + (MODE == MODE_FC1 ? p.I + col0 : col0 + 32));
          float w0[32], w1[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 a4 = __ldg(c0 + i), b4 = __ldg(c1 + i);
            w0[4 * i] = a4.x; w0[4 * i + 1] = a4.y; w0[4 * i + 2] = a4.z; w0[4 * i + 3] = a4.w;
            w1[4 * i] = b4.x; w1[4 * i + 1] = b4.y; w1[4 * i + 2] = b4.z; w1[4 * i + 3] = b4.w;
          }
          if (MODE == MODE_FC1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float g = (rs * w0[i]) * s0[i];
              const float u = (rs * w1[i]) * s1[i];
              pk[i] = __float_as_uint(silu_f(g) * u);
            }
          } else {  // y as fp16 with a power-of-two scale per 64 columns
            uint32_t y0[32], y1[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              y0[i] = __float_as_uint((rs * w0[i]) * s0[i]);
              y1[i] = __float_as_uint((rs * w1[i]) * s1[i]);
            }
            const float inv = pack_y16(y0, y1, pk);
            if (valid) p.yscale[static_cast<int64_t>(grow) * (p.H / 64) + col0 / 64] = inv;
          }
          const int out_cols = MODE == MODE_FC1 ? p.I : p.H;
          constexpr int ESZ = MODE == MODE_FC1 ? 4 : 2;   // h fp32, y fp16
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<uint4*>(stage + row_off + ((v ^ (lane & 7)) << 4)) =
                make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          if (wrows == 32) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOut, stage, col0, grow0);
              bulk_commit();
            }
          } else if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(p.out) +
                                                  (static_cast<int64_t>(grow) * out_cols + col0) * ESZ);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = *reinterpret_cast<const uint4*>(stage + row_off + ((v ^ (lane & 7)) << 4));
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfree[F]);  // slot F read (after tcgen05.wait::ld)
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// int8 -> bf16 (exact), 16 values per thread step, over one or two tensors
// (one launch: segment 0 then segment 1 in one grid-stride range)
__global__ void i8_to_bf16_kernel(const int8_t* __restrict__ src0, __nv_bfloat16* __restrict__ dst0,
                                  size_t n16_0, const int8_t* __restrict__ src1,
                                  __nv_bfloat16* __restrict__ dst1, size_t n16_1) {
  griddep_wait();
  griddep_launch_dependents();
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (; i < n16_0 + n16_1; i += stride) {
    const bool first = i < n16_0;
    const size_t j = first ? i : i - n16_0;
    const int4 v = __ldg(reinterpret_cast<const int4*>(first ? src0 : src1) + j);
    const int8_t* b = reinterpret_cast<const int8_t*>(&v);
    uint32_t w[8];
#pragma unroll
    for (int t = 0; t < 8; ++t)
      w[t] = pack_bf16x2(static_cast<float>(b[2 * t]), static_cast<float>(b[2 * t + 1]));
    uint4* d = reinterpret_cast<uint4*>(first ? dst0 : dst1) + 2 * j;
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// Symmetric per-row int8 re-quantisation of h (one warp per permuted row):
// hs = max|h| / 127 (1 for an all-zero row), hq = rne(h / hs) clamped to
// [-127, 127]; IEEE division, as a float32 program would do it.
__global__ void requant_rows_kernel(const float* __restrict__ h, const int32_t* __restrict__ offsets,
                                    int E, int I, int8_t* __restrict__ hq, float* __restrict__ hs) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  griddep_wait();
  griddep_launch_dependents();
  if (row >= __ldg(offsets + E)) return;
  const float4* hr = reinterpret_cast<const float4*>(h + row * I);
  float m = 0.f;
  for (int c = lane; c < I / 4; c += 32) {
    const float4 v = __ldg(hr + c);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float scale = m > 0.f ? __fdiv_rn(m, 127.0f) : 1.0f;
  if (lane == 0) hs[row] = scale;
  char4* qr = reinterpret_cast<char4*>(hq + row * I);
  for (int c = lane; c < I / 4; c += 32) {
    const float4 v = __ldg(hr + c);
    auto q = [&](float x) {
      const float r = rintf(__fdiv_rn(x, scale));
      return static_cast<signed char>(fminf(fmaxf(r, -127.f), 127.f));
    };
    qr[c] = make_char4(q(v.x), q(v.y), q(v.z), q(v.w));
  }
}

// The same with the row held in registers (NV float4 per lane, I <= 128 NV):
// one read of h, every load of the row in flight before the max.
template <int NV>
__global__ void requant_rows_reg_kernel(const float* __restrict__ h,
                                        const int32_t* __restrict__ offsets, int E, int I,
                                        int8_t* __restrict__ hq, float* __restrict__ hs) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  griddep_wait();
  griddep_launch_dependents();
  if (row >= __ldg(offsets + E)) return;
  const int I4 = I / 4;
  const float4* hr = reinterpret_cast<const float4*>(h + row * I);
  float4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = lane + 32 * i;
    v[i] = c < I4 ? __ldg(hr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i)
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float scale = m > 0.f ? __fdiv_rn(m, 127.0f) : 1.0f;
  if (lane == 0) hs[row] = scale;
  char4* qr = reinterpret_cast<char4*>(hq + row * I);
  auto q = [&](float x) {
    const float r = rintf(__fdiv_rn(x, scale));
    return static_cast<signed char>(fminf(fmaxf(r, -127.f), 127.f));
  };
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = lane + 32 * i;
    if (c < I4) qr[c] = make_char4(q(v[i].x), q(v[i].y), q(v[i].z), q(v[i].w));
  }
}

cudaError_t launch_i8_to_bf16_2(const int8_t* src0, void* dst0, size_t n0, const int8_t* src1,
                                void* dst1, size_t n1, cudaStream_t st) {
  // every int8 tensor converted here has a multiple of 64 elements
  const size_t n16_0 = n0 / 16, n16_1 = n1 / 16;
  if (n16_0 + n16_1 == 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = static_cast<unsigned>(
      std::min<size_t>((n16_0 + n16_1 + threads - 1) / threads, 152 * 32));
  const cudaError_t e =
      launch_kernel(i8_to_bf16_kernel, dim3(blocks), dim3(threads), 0, st, 1, src0,
                    static_cast<__nv_bfloat16*>(dst0), n16_0, src1,
                    static_cast<__nv_bfloat16*>(dst1), n16_1);
  note_launches(1);
  return e;
}

cudaError_t launch_i8_to_bf16(const int8_t* src, void* dst, size_t n, cudaStream_t st) {
  return launch_i8_to_bf16_2(src, dst, n, nullptr, nullptr, 0, st);
}

cudaError_t launch_requant(const float* h, const int32_t* offsets, const mc2_shape_t& s, int8_t* hq,
                           float* hs, cudaStream_t st) {
  const int64_t R = static_cast<int64_t>(s.T) * s.k;
  if (R == 0) return cudaSuccess;
  const int warps = 8;
  const dim3 grid(static_cast<unsigned>((R + warps - 1) / warps)), block(warps * 32);
  const int E = static_cast<int>(s.E), I = static_cast<int>(s.I);
  cudaError_t e;
  if (I <= 512)
    e = launch_kernel(requant_rows_reg_kernel<4>, grid, block, 0, st, 1, h, offsets, E, I, hq, hs);
  else if (I <= 1024)
    e = launch_kernel(requant_rows_reg_kernel<8>, grid, block, 0, st, 1, h, offsets, E, I, hq, hs);
  else if (I <= 1536)
    e = launch_kernel(requant_rows_reg_kernel<12>, grid, block, 0, st, 1, h, offsets, E, I, hq, hs);
  else if (I <= 2048)
    e = launch_kernel(requant_rows_reg_kernel<16>, grid, block, 0, st, 1, h, offsets, E, I, hq, hs);
  else
    e = launch_kernel(requant_rows_kernel, grid, block, 0, st, 1, h, offsets, E, I, hq, hs);
  note_launches(1);
  return e;
}

template <int MODE, bool PAIR>
static cudaError_t launch_q(const QArgs& g, cudaStream_t st) {
  const mc2_shape_t& s = *g.s;
  const int64_t R = static_cast<int64_t>(s.T) * s.k;
  CUtensorMap tA, tB, tOut;
  QParams p;
  p.a_ptr = g.a;
  p.offsets = g.offsets;
  p.permute_src = g.permute_src;
  p.a_scale = g.a_scale;
  p.b_scale = g.b_scale;
  p.out = g.out;
  p.yscale = g.yscale;
  p.dev_status = g.dev_status;
  p.E = s.E;
  p.k = s.k;
  p.I = s.I;
  p.H = s.H;
  p.raw = g.raw ? 1 : 0;
  p.wait_limit_ns = wait_limit_ns();
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  bool ok;
  if (MODE == MODE_FC1) {
    p.K = s.H;
    p.n_tiles = s.I / 64;
    ok = encode_b_blocked(&tB, g.b, s.H, 2ull * s.I, s.E, 2, 64, 1, PAIR ? 1 : 2);
    tA = tB;  // unused: fc1's A rows are gathered with cp.async
    tOut = tB;
    if (!g.raw) ok = ok && encode_2d(&tOut, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.out, s.I, R, 32, 32);
  } else {
    p.K = s.I;
    p.n_tiles = (s.H + QBN - 1) / QBN;  // H is a multiple of 64: the last tile may be half full
    ok = encode_2d(&tA, bf, 2, g.a, s.I, R, 64, BM) &&
         encode_b_blocked(&tB, g.b, s.I, s.H, s.E, 1, 64, PAIR ? 1 : 2, 1);
    tOut = tB;
    if (!g.raw) ok = ok && encode_2d(&tOut, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.out, s.H, R, 64, 32);
  }
  if (!ok) return cudaErrorInvalidValue;
  p.nchunk = (p.K / 64 + QCHUNK_KB - 1) / QCHUNK_KB;
  if (p.nchunk > QMAX_CHUNKS) return cudaErrorInvalidValue;
  using G = QGeom<PAIR>;
  const size_t smem = G::kSmemFixed + (s.E + 1) * sizeof(int32_t);
  static PerDevice<KernelSetup> setup;
  const KernelSetup su = once_per_device(setup, [] {
    return setup_kernel(gmm_q_kernel<MODE, PAIR>, G::kSmemFixed + 1025 * sizeof(int32_t),
                        QRoles<MODE>::kThreads, PAIR);
  });
  if (su.err != cudaSuccess) return su.err;
  const int max_clusters = su.pair_clusters;
  if (PAIR) {  // persistent grid: as many pairs as can be resident at once
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    const int64_t tiles_upper = (R / (2 * BM) + s.E) * static_cast<int64_t>(p.n_tiles);
    const int grid =
        2 * static_cast<int>(std::min<int64_t>(max_clusters, std::max<int64_t>(tiles_upper, 1)));
    return launch_kernel(gmm_q_kernel<MODE, PAIR>, dim3(grid), dim3(QRoles<MODE>::kThreads), smem,
                         st, 2, tA, tB, tOut, p);
  }
  const int64_t tiles_upper = (R / BM + s.E) * static_cast<int64_t>(p.n_tiles);
  const int grid = static_cast<int>(std::min<int64_t>(num_sms(), std::max<int64_t>(tiles_upper, 1)));
  return launch_kernel(gmm_q_kernel<MODE, PAIR>, dim3(grid), dim3(QRoles<MODE>::kThreads), smem,
                       st, 1, tA, tB, tOut, p);
}

template <int MODE>
static cudaError_t launch_qw(const QArgs& g, cudaStream_t st) {
  const mc2_shape_t& s = *g.s;
  const int64_t R = static_cast<int64_t>(s.T) * s.k;
  CUtensorMap tA, tB, tOut;
  QParams p;
  p.a_ptr = g.a;
  p.offsets = g.offsets;
  p.permute_src = g.permute_src;
  p.a_scale = g.a_scale;
  p.b_scale = g.b_scale;
  p.out = g.out;
  p.yscale = g.yscale;
  p.dev_status = g.dev_status;
  p.E = s.E;
  p.k = s.k;
  p.I = s.I;
  p.H = s.H;
  p.raw = g.raw ? 1 : 0;
  p.wait_limit_ns = wait_limit_ns();
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  bool ok;
  if (MODE == MODE_FC1) {
    p.K = s.H;
    p.n_tiles = (s.I + 127) / 128;  // I is a multiple of 64: the last tile may be half full
    ok = encode_b_blocked(&tB, g.b, s.H, 2ull * s.I, s.E, 2, 64, 2, 2);
    tA = tB;  // unused: fc1's A rows are gathered with cp.async
    tOut = tB;
    if (!g.raw) ok = ok && encode_2d(&tOut, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.out, s.I, R, 32, 32);
  } else {
    p.K = s.I;
    p.n_tiles = (s.H + QW_BN - 1) / QW_BN;
    ok = encode_2d(&tA, bf, 2, g.a, s.I, R, 64, BM) &&
         encode_b_blocked(&tB, g.b, s.I, s.H, s.E, 1, 64, 4, 1);
    tOut = tB;
    if (!g.raw) ok = ok && encode_2d(&tOut, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.out, s.H, R, 64, 32);
  }
  if (!ok) return cudaErrorInvalidValue;
  p.nchunk = (p.K / 64 + QCHUNK_KB - 1) / QCHUNK_KB;
  if (p.nchunk > QMAX_CHUNKS) return cudaErrorInvalidValue;
  const size_t smem = QW_SMEM_FIXED + (s.E + 1) * sizeof(int32_t);
  static PerDevice<KernelSetup> setup;
  const KernelSetup su = once_per_device(setup, [] {
    return setup_kernel(gmm_qw_kernel<MODE>, QW_SMEM_FIXED + 1025 * sizeof(int32_t),
                        QRoles<MODE>::kThreads, false);
  });
  if (su.err != cudaSuccess) return su.err;
  const int64_t tiles_upper = (R / BM + s.E) * static_cast<int64_t>(p.n_tiles);
  const int grid = static_cast<int>(std::min<int64_t>(num_sms(), std::max<int64_t>(tiles_upper, 1)));
  return launch_kernel(gmm_qw_kernel<MODE>, dim3(grid), dim3(QRoles<MODE>::kThreads), smem, st, 1,
                       tA, tB, tOut, p);
}

// Tiling of the int8 GEMMs (every form gives the same bits: each output
// accumulates its chunks in the same K order and is dequantised alike):
// by default the wide single-CTA kernel (128 x 256 tiles); mc2_set_tile_pairing
// 1 selects the 128 x 128 single-CTA kernel, 2 the 256 x 128 CTA pairs.
// Measured on GB300 with the 8192-token int8 workload (about 512 rows per
// expert), 128 x 128 against pairs: block 1.509 vs 1.736 ms (256-row tiles
// pad more rows, and fc1's odd CTA relays its gathered stages).
cudaError_t launch_gemm_q(const QArgs& g, cudaStream_t st) {
  if (static_cast<int64_t>(g.s->T) * g.s->k == 0) return cudaSuccess;
  const int forced = tile_pairing_override();
  cudaError_t e;
  if (forced == 2 && num_sms() >= 2)
    e = g.mode == MODE_FC1 ? launch_q<MODE_FC1, true>(g, st) : launch_q<MODE_FC2, true>(g, st);
  else if (forced == 1)
    e = g.mode == MODE_FC1 ? launch_q<MODE_FC1, false>(g, st) : launch_q<MODE_FC2, false>(g, st);
  else
    e = g.mode == MODE_FC1 ? launch_qw<MODE_FC1>(g, st) : launch_qw<MODE_FC2>(g, st);
  note_launches(1);
  return e;
}

}  // namespace mc2
