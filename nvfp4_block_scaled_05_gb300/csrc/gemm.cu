// Persistent NVFP4 grouped GEMM for sm_103a ("NVFP4 MegaMoE Kernel" README,
// "ScaledGroupedGemmKernel": A(M,K) x B(E,K,N) -> C(M,N), block-scaled on both
// operands, per-expert global scales, persistent scheduler, TMA pipelining,
// swizzled shared memory; and "Fused SwiGLU - How It Works" for the L1
// epilogue, extended with "Remaining Steps" 2-4: NVFP4 requantization in the
// epilogue, FP4 codes and scales stored straight into the padded L2 input).
//
// Tile: 128 activation rows (one expert) x 256 weight rows, one
// tcgen05.mma kind::mxf4nvf4 (M=128, N=256, K=64) per 64 K; K streamed in
// stages of 256 elements (one 128-byte swizzle row per operand row).
// Measured on this part: an M=128 MMA costs the same issue time for N=64..256,
// so N=256 is the shape that reaches the tensor-core rate. The block scales
// must sit in tensor memory before each MMA; moving them with tcgen05.cp
// (about 35 bytes of TMEM per cycle, one copy engine) costs more than the MMAs
// it feeds, so four warps write them with tcgen05.st instead, each into its
// own TMEM lane quadrant, in parallel.
// Warp roles (480 threads, one CTA per SM):
//   warp 0      TMA producer: A and B code tiles (tiled TMA, 128B swizzle)
//               into a 4-stage ring
//   warp 1      TMEM owner; one lane issues the MMAs
//   warps 2-5   scale warps, one per TMEM lane quadrant q: per stage, once the
//               stage's scale atoms have landed, the A scale of each of the
//               quadrant's 32 rows goes to column 4kk+q for K=64 step kk (the
//               MMA reads quadrant q's A scales from column base+q), and the
//               256 B-row scales to columns 8kk..8kk+7 (B scales are read in
//               every quadrant, so each quadrant holds its own copy)
//   warps 6-13  epilogue, two warps per TMEM lane quadrant (128 columns
//               each): the f32 accumulator is moved to registers and released
//               (L1: the first 64 columns become h before the second 64 are
//               loaded), so the next tile's MMAs overlap the epilogue math;
//               then BF16 output (L2, streaming stores) or SwiGLU + NVFP4
//               requant (L1, h in the row-tiled scale layout the L2 GEMM reads)
//   warp 14     one lane issues the scale atoms' bulk copies (activation:
//               128 rows x 16 bytes, row-tiled layout; weights: 512-byte
//               atoms) of each stage into its scale slot, after the same wait
//               for a free stage as the producer. Per stage the load round trip
//               (slot free -> copies issued -> landed -> MMAs -> slot free)
//               bounds the kernel, and issuing five copies from one thread put
//               ~640 cycles of it on every stage; with the scale copies here
//               the producer spends ~160.
// Tiles are ordered expert-major, then weight tile, then activation tile, so
// the activation tiles sharing one weight tile run at the same time on
// neighbouring SMs and the weight tile leaves HBM once.
//
// 2-SM pairs (kPair, opt-in): a cluster of two CTAs on one tile of 256
// activation rows (the even CTA's 128, then the odd CTA's) x 256 weight rows;
// each CTA loads its activation rows and half of the weight rows, and the even
// CTA issues tcgen05.mma.cta_group::2 (M=256) whose result rows land in each
// CTA's own tensor memory. Both CTAs' code tiles complete on the even CTA's
// stage barrier (the pair form of the tensor copy), both CTAs' scale warps and
// epilogues arrive on the even CTA's barriers, so the MMA issuer waits once
// per stage as in the one-CTA kernel; the MMA commits arrive on both CTAs'
// barriers.
//
// Every wait is bounded: a wait that exceeds the limit sets the device status
// word, raises a shared abort flag that ends the other roles' loops, and the
// CTA then waits (with a fixed bound) for its own copies and tensor-core work
// in flight, frees its tensor memory and returns.
#include "common.cuh"

namespace nvfp4moe {

__device__ int g_status[2];  // [0]: NVFP4MOE_OK or NVFP4MOE_ERR_DEVICE_TIMEOUT, [1]: wait site

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 256;                       // K elements per stage
constexpr int kScaleWarps = 4;
constexpr int kEpiWarps = 8;
constexpr int kFirstEpiWarp = 2 + kScaleWarps;
constexpr int kCopyWarp = kFirstEpiWarp + kEpiWarps;   // issues the scale atoms' bulk copies
constexpr int kThreads = 32 * (kCopyWarp + 1);
constexpr int A_BYTES = BM * BK / 2;          // 16 KB
constexpr int SFA_BYTES = 4 * 512;            // 4 scale atoms (K=256) of 128 rows
constexpr int SF_BYTES = 3 * SFA_BYTES;       // SFA, then SFB's two 128-row halves
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = BN;             // one f32 accumulator of 256 columns
constexpr uint32_t SFB_SLOT = 32;
constexpr uint32_t SFA_SLOT = 16;
constexpr uint64_t kDrainLimitNs = 1000000000ull;
constexpr uint64_t kPairCopyDrainNs = 2000000ull;   // 2 ms

// Shared- and tensor-memory plan of one CTA. kPair: the CTA is one half of a
// 2-SM pair and holds only its 128 of the tile's 256 weight rows, which frees
// shared memory for a fifth stage.
template <bool kPair>
struct Cfg {
  static constexpr int STAGES = kPair ? 5 : 4;
  static constexpr int B_ROWS = kPair ? BN / 2 : BN;    // weight rows this CTA loads per tile
  static constexpr int B_BYTES = B_ROWS * BK / 2;       // 16 / 32 KB
  static constexpr int OFF_B = STAGES * A_BYTES;
  static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = OFF_SF + STAGES * SF_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + (kPair ? 512 : 256);
  static constexpr int OFF_SCHED = OFF_MISC + 256;
  // Scale slots after the accumulator. A TMEM store of n columns starts on a
  // multiple of n, so each stage's 32 SFB columns (k-step kk in columns 8kk ..
  // 8kk+7) start on a multiple of 32, and the SFA slots (quadrant q: k-step kk
  // in column 4kk + q, one-column stores) follow all of them.
  static constexpr uint32_t SFB_TMEM0 = ACC_COLS;
  static constexpr uint32_t SFA_TMEM0 = SFB_TMEM0 + STAGES * SFB_SLOT;
  static_assert(SFA_TMEM0 + STAGES * SFA_SLOT <= TMEM_COLS, "tensor memory budget");
  static_assert(OFF_SCHED + 8 * 1025 + 1024 <= 232448, "shared memory budget");
  static_assert((kPair ? 3 * STAGES + 5 : 3 * STAGES + 4) * 8 <= OFF_MISC - OFF_BAR, "barrier area");
};

struct Params {
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  const float* gs_a;
  const float* gs_b;
  const int32_t* offsets;
  int E;
  int N;
  int K;
  int64_t sf_rowtile_bytes;   // (K/64) * 512: weight scale bytes of 128 rows (NVFP4_SF_TILED)
  int64_t a_sf_rowtile_bytes; // ceil(K/256) * 2048: activation scale bytes of 128 rows (TILED_ROWS)
  int64_t b_sf_expert_bytes;  // scale bytes of one expert's N x K weights
  // plain epilogue
  __nv_bfloat16* c;
  int64_t ldc;
  int c_32B;                  // c and ldc allow 32-byte stores
  // SwiGLU epilogue
  uint8_t* h_codes;
  uint8_t* h_sf;
  int64_t I;
  const float* gs_h;
  uint64_t wait_limit_ns;
  int* status;
  int test_stall;             // test hook: the MMA issuer first waits on a barrier nobody arrives on
};

// Work units, ordered expert-major, then weight tile, then activation tile(s).
// A unit is one 128-row activation tile x one 256-row weight tile, or with
// pairs two consecutive activation tiles of the expert (the even CTA takes the
// first, the odd CTA the second, which may not exist) x one weight tile.
struct Sched {
  const int32_t* tile_start;  // [E+1] first unit of each expert
  const int32_t* pad_off;     // [E+1] padded first row of each expert
  const int32_t* offsets;     // [E+1] compact first row of each expert
  int E;
  int NT;                     // weight tiles per expert
  int N;
  int pair;                   // 1: units of two activation tiles
  // rows <= 0: no activation tile of this CTA in the unit (the odd CTA of a
  // pair whose expert has an odd number of activation tiles)
  __device__ __forceinline__ void decode(int t, int rank, int& e, int& nb, int& mb, int& rows, int& ncols) const {
    int lo = 0, hi = E - 1;
    while (lo < hi) {  // largest e with tile_start[e] <= t
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    const int per = (tile_start[e + 1] - tile_start[e]) / NT;   // units per weight tile
    const int local = t - tile_start[e];
    nb = local / per;
    const int m = local - nb * per;
    mb = pair ? 2 * m + rank : m;
    const int cnt = offsets[e + 1] - offsets[e];
    rows = min(BM, cnt - mb * BM);
    ncols = min(BN, N - nb * BN);   // 256, or 128 for the last tile when N % 256 == 128
  }
};

// Bounded wait. Returns false on timeout (after raising the abort flag, the
// pair peer's abort flag when peer_abort != 0, and the device status) or when
// another role has aborted. kCluster: the barrier is arrived on from the pair
// peer (acquire at cluster scope).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             uint64_t limit_ns, int* status, int site, uint32_t peer_abort = 0) {
  auto probe = [&]() { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (probe()) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (probe()) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        if (peer_abort) st_shared_cluster_u32(peer_abort, 1u);
        if (atomicCAS(&status[0], 0, NVFP4MOE_ERR_DEVICE_TIMEOUT) == 0) status[1] = site;
        return false;
      }
    }
  }
}

// Wait used while shutting down: ignores the abort flag, fixed bound.
template <bool kCluster = false>
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!(kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity))) {
    if (global_timer_ns() - t0 > kDrainLimitNs) return;
  }
}

// silu(g) = g / (1 + exp(-g)) with the hardware exponential and reciprocal
// (a few ulp; h is requantized to 4 bits right after).
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

template <bool kSwiGLU, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a16,
                        const __grid_constant__ CUtensorMap tm_a32,
                        const __grid_constant__ CUtensorMap tm_a64,
                        const __grid_constant__ CUtensorMap tm_a128,
                        const __grid_constant__ CUtensorMap tm_b, const Params p) {
  using C = Cfg<kPair>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(smem);
  // full[s]: stage s's code tiles landed (the producer's expect_tx) and its
  // scales are in tensor memory (one arrival per scale warp): the one barrier
  // the MMA issuer waits on per stage (every wait in its loop costs the tensor
  // pipe; measured, the per-stage waits were ~11% of a load-free MMA stream)
  const uint32_t bar_full = sbase + C::OFF_BAR;            // STAGES x 8 bytes each
  const uint32_t bar_empty = bar_full + STAGES * 8;
  const uint32_t bar_accf = bar_empty + STAGES * 8;
  const uint32_t bar_acce = bar_accf + 8;
  const uint32_t bar_aux = bar_acce + 8;                   // MMA drain on abort
  const uint32_t bar_never = bar_aux + 8;                  // never arrived on (failure-path test)
  const uint32_t bar_sffull = bar_never + 8;               // STAGES: a stage's scale atoms landed
  // pairs: the exit handshake
  const uint32_t bar_exit = bar_sffull + STAGES * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int32_t* tile_start = reinterpret_cast<int32_t*>(smem + C::OFF_SCHED);
  int32_t* pad_off = tile_start + (p.E + 1);
  const int E = p.E, NT = (p.N + BN - 1) / BN;
  // pairs: rank 0 (the even CTA) issues the MMAs of both
  const int rank = kPair ? (int)cluster_ctarank() : 0;
  const int first_unit = kPair ? (int)blockIdx.x / 2 : (int)blockIdx.x;
  const int unit_stride = kPair ? (int)gridDim.x / 2 : (int)gridDim.x;
  const uint32_t peer_abort = kPair ? mapa_shared(smem_addr(smem + C::OFF_MISC + 4), rank ^ 1) : 0u;
  // pairs: the even CTA's full barriers (both CTAs' code tiles complete on
  // them and both CTAs' scale warps arrive on them) and accumulator-empty
  // barrier (both CTAs' epilogues arrive on it), as shared::cluster addresses
  const uint32_t pair_full0 = kPair ? mapa_shared(bar_full, 0) : 0u;
  const uint32_t pair_acce = kPair ? mapa_shared(bar_acce, 0) : 0u;

  // --- schedule: per expert its units (ceil(n_e/128) activation tiles, or
  //     ceil of half of that with pairs, per weight tile), prefix sums
  if (warp == 0) {
    int carry = 0, carry_rows = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int mt = e < E ? (p.offsets[e + 1] - p.offsets[e] + BM - 1) / BM : 0;
      const int mu = kPair ? (mt + 1) / 2 : mt;
      int incl = mu, incl_rows = mt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        const int yr = __shfl_up_sync(0xFFFFFFFFu, incl_rows, d);
        if (lane >= d) {
          incl += y;
          incl_rows += yr;
        }
      }
      if (e < E) {
        tile_start[e] = (carry + incl - mu) * NT;
        pad_off[e] = (carry_rows + incl_rows - mt) * BM;
      }
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
      carry_rows += __shfl_sync(0xFFFFFFFFu, incl_rows, 31);
    }
    if (lane == 0) {
      tile_start[E] = carry * NT;
      pad_off[E] = carry_rows * BM;
    }
  }
  if (tid == 32) {
    for (int s = 0; s < STAGES; ++s) {
      // pairs (used in the even CTA only): the even producer's expect_tx and
      // the scale warps of both CTAs
      mbar_init(bar_full + 8 * s, 1 + kScaleWarps * (kPair ? 2 : 1));
      mbar_init(bar_sffull + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_accf, 1);
    // every epilogue thread of this CTA; pairs: and one lane per epilogue warp
    // of the odd CTA
    mbar_init(bar_acce, kEpiWarps * 32 + (kPair ? kEpiWarps : 0));
    mbar_init(bar_aux, 1);
    mbar_init(bar_never, 1);
    if constexpr (kPair) mbar_init(bar_exit, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_addr(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (kPair) cluster_sync_all();   // the peer's barriers exist before anyone arrives on them
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = tile_start[E];
  const Sched sch{tile_start, pad_off, p.offsets, E, NT, p.N, kPair ? 1 : 0};
  const int ksteps = p.K / 64;
  const int kblocks = (ksteps + 3) / 4;
  const int my_units = first_unit < total ? (total - 1 - first_unit) / unit_stride + 1 : 0;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- producer
    prefetch_tensormap(&tm_a16);
    prefetch_tensormap(&tm_a32);
    prefetch_tensormap(&tm_a64);
    prefetch_tensormap(&tm_a128);
    prefetch_tensormap(&tm_b);
    // Weights: a weight tile read by one unit is streamed once (evict first);
    // one that several units of a large expert read in turn keeps normal
    // priority, so that the activation and output streams do not push it out
    // of L2 before its last reader.
    const uint64_t pol_w1 = l2_policy_evict_first();
    const uint64_t pol_wn = l2_policy_evict_normal();
    const uint64_t pol_a = l2_policy_evict_last();   // activations: reused by every weight tile
    // Copy sources of one unit's code tiles, decoded one unit ahead of its loads.
    // pairs: tx_bytes also counts the odd CTA's tiles (the even CTA arms the
    // barrier both CTAs' copies complete on)
    struct TileSrc {
      const CUtensorMap* tma;
      int box, a_row, b_row;
      uint32_t tx_bytes;
      bool has_a;
      uint64_t pol_w;
    };
    auto a_box = [](int rows) { return rows <= 0 ? 0 : rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128; };
    auto tile_src = [&](int t) {
      int e, nb, mb, rows, ncols;
      sch.decode(t, rank, e, nb, mb, rows, ncols);
      TileSrc c;
      c.pol_w = tile_start[e + 1] - tile_start[e] > NT ? pol_wn : pol_w1;
      c.has_a = rows > 0;
      c.tma = rows <= 16 ? &tm_a16 : rows <= 32 ? &tm_a32 : rows <= 64 ? &tm_a64 : &tm_a128;
      c.box = a_box(rows);
      c.a_row = pad_off[e] + mb * BM;
      c.b_row = e * p.N + nb * BN + rank * C::B_ROWS;
      c.tx_bytes = (uint32_t)(c.box * 128 + C::B_ROWS * 128);
      if constexpr (kPair) {
        if (rank == 0) {
          int e1, nb1, mb1, rows1, ncols1;
          sch.decode(t, 1, e1, nb1, mb1, rows1, ncols1);
          c.tx_bytes += (uint32_t)(a_box(rows1) * 128 + C::B_ROWS * 128);
        }
      }
      return c;
    };
    uint32_t stage = 0, phase = 0, filled = 0, fill_phase = 0;
    bool ok = true;
    TileSrc cur{}, nxt{};
    if (first_unit < total) cur = tile_src(first_unit);
    for (int t = first_unit; ok && t < total; t += unit_stride) {
      const bool has_next = t + unit_stride < total;
      if (has_next) nxt = tile_src(t + unit_stride);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_bounded(bar_empty + 8 * stage, phase ^ 1, abort_flag, p.wait_limit_ns, p.status, 1, peer_abort)) {
          ok = false;
          break;
        }
        // the B box always moves B_ROWS rows; rows past this expert's last
        // weight tile are never multiplied (N=128 MMA), rows past the tensor
        // read zeros
        if constexpr (kPair) {
          // both CTAs' tiles complete on the even CTA's barrier, which only
          // the even CTA arms (a copy may land before it is armed: the phase
          // cannot complete while the arrival is missing)
          const uint32_t full = pair_full0 + 8 * stage;
          if (rank == 0) mbar_arrive_expect_tx(bar_full + 8 * stage, cur.tx_bytes);
          if (cur.has_a) tma_load_2d_pair(sbase + stage * A_BYTES, cur.tma, full, kb * 128, cur.a_row, pol_a);
          tma_load_2d_pair(sbase + C::OFF_B + stage * C::B_BYTES, &tm_b, full, kb * 128, cur.b_row, cur.pol_w);
        } else {
          const uint32_t full = bar_full + 8 * stage;
          mbar_arrive_expect_tx(full, cur.tx_bytes);
          if (cur.has_a) tma_load_2d(sbase + stage * A_BYTES, cur.tma, full, kb * 128, cur.a_row, pol_a);
          tma_load_2d(sbase + C::OFF_B + stage * C::B_BYTES, &tm_b, full, kb * 128, cur.b_row, cur.pol_w);
        }
        filled |= 1u << stage;
        fill_phase = (fill_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      cur = nxt;
    }
    if (!ok) {
      // copies still in flight complete before the CTA may exit. A pair's
      // copies complete on the even CTA's barriers together with the other
      // CTA's, whose producer may have stopped before arming or issuing its
      // part, so a pair waits a fixed time instead: far longer than a copy
      // takes to land (microseconds), and both CTAs then still pass the exit
      // handshake, so neither leaves while the other's copies may land.
      if constexpr (kPair) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < kPairCopyDrainNs) {
        }
      } else {
        for (int s = 0; s < STAGES; ++s)
          if ((filled >> s) & 1u) drain_wait(bar_full + 8 * s, (fill_phase >> s) & 1u);
      }
    } else if constexpr (kPair) {
      // every stage's last use released by the even CTA's MMAs (whose commits
      // arrive on this CTA's barriers) before the CTA may exit
      for (int i = 0; i < STAGES; ++i) {
        if (!wait_bounded(bar_empty + 8 * stage, phase ^ 1, abort_flag, p.wait_limit_ns, p.status, 10, peer_abort))
          break;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp == kCopyWarp && lane == 0) {
    // ---------------------------------------------------------------- scale copies
    // The scale atoms of each stage (activation: 128 rows x 16 bytes, 2048
    // bytes whatever the K tail; weights: the 512-byte atoms of the tile's two
    // 128-row halves) as bulk copies into the stage's scale slot, once the
    // stage is free (the same wait as the producer's). A thread of its own, so
    // that the producer issues only the two code tiles per stage: each copy
    // costs its issuing thread ~130 cycles, and with all five on one thread
    // that issue time sat on the load round trip of every stage.
    const uint64_t pol_a = l2_policy_evict_last();
    const uint64_t pol_w1 = l2_policy_evict_first();
    const uint64_t pol_wn = l2_policy_evict_normal();
    uint32_t stage = 0, phase = 0, filled = 0, fill_phase = 0;
    bool ok = true;
    for (int t = first_unit; ok && t < total; t += unit_stride) {
      int e, nb, mb, rows, ncols;
      sch.decode(t, rank, e, nb, mb, rows, ncols);
      const bool has_a = rows > 0;
      const uint64_t pol_w = tile_start[e + 1] - tile_start[e] > NT ? pol_wn : pol_w1;
      const uint8_t* sfa = p.a_sf + (int64_t)((pad_off[e] + mb * BM) / BM) * p.a_sf_rowtile_bytes;
      const uint8_t* sfb = p.b_sf + (int64_t)e * p.b_sf_expert_bytes + (int64_t)(nb * 2) * p.sf_rowtile_bytes;
      const int bhalves = ncols / 128;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_bounded(bar_empty + 8 * stage, phase ^ 1, abort_flag, p.wait_limit_ns, p.status, 16, peer_abort)) {
          ok = false;
          break;
        }
        const int nk = min(4, ksteps - kb * 4);
        const uint32_t sffull = bar_sffull + 8 * stage;
        const uint32_t sdst = sbase + C::OFF_SF + stage * SF_BYTES;
        mbar_arrive_expect_tx(sffull, (has_a ? 2048 : 0) + bhalves * nk * 512);
        if (has_a) bulk_load(sdst, sfa + kb * 2048, 2048, sffull, pol_a);
        for (int h = 0; h < bhalves; ++h)
          bulk_load(sdst + SFA_BYTES + h * SFA_BYTES, sfb + h * p.sf_rowtile_bytes + kb * 2048, nk * 512, sffull,
                    pol_w);
        filled |= 1u << stage;
        fill_phase = (fill_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok)   // copies still in flight complete before the CTA may exit
      for (int s = 0; s < STAGES; ++s)
        if ((filled >> s) & 1u) drain_wait(bar_sffull + 8 * s, (fill_phase >> s) & 1u);
  } else if (warp >= 2 && warp < kFirstEpiWarp) {
    // ---------------------------------------------------------------- scale warps
    // Per stage, each warp stores its quadrant's scales into the stage's TMEM
    // slot once the stage's atoms have landed (the slot's previous MMAs are
    // done by then: the copies were issued after them). A pair CTA without an
    // activation tile in the unit stores zero A scales (its rows of the MMA
    // are discarded).
    const int q = warp & 3;                               // TMEM lane quadrant of this warp
    const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
    const int nstages = my_units * kblocks;
    bool ok = true;
    bool use_has_a = true;                                // the consumed unit has this CTA's activation tile
    int g = 0;
    for (; ok && g < nstages; ++g) {
      if constexpr (kPair) {
        if (g % kblocks == 0) {
          int e, nb, mb, rows, ncols;
          sch.decode(first_unit + (g / kblocks) * unit_stride, rank, e, nb, mb, rows, ncols);
          use_has_a = rows > 0;
        }
      }
      const int slot = g % STAGES, use = g / STAGES;
      ok = wait_bounded(bar_sffull + 8 * slot, use & 1, abort_flag, p.wait_limit_ns, p.status, 5, peer_abort);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      // Activation scales: row r's 16 blocks are the 16 bytes at r * 16, the
      // word of k-step kk at r * 16 + 4 kk. Weight atoms: 16-byte chunk `lane`
      // of a 512-byte atom holds rows lane, lane+32, lane+64, lane+96 (4 bytes
      // each, one per 16-element block). Slots past a K tail (and the second
      // half of a 128-column tile) hold stale bytes the MMAs never read.
      const uint8_t* ssfa = smem + C::OFF_SF + slot * SF_BYTES + (q * 32 + lane) * 16;
      const uint8_t* ssfb = smem + C::OFF_SF + slot * SF_BYTES + SFA_BYTES + lane * 16;
      uint32_t a[4], b[32];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        a[kk] = use_has_a ? *reinterpret_cast<const uint32_t*>(ssfa + kk * 4) : 0u;   // row 32q + lane
        // B rows lane+32j, j = 0..3 (first 128 rows) and 4..7 (second 128 rows)
        const uint4 lo = *reinterpret_cast<const uint4*>(ssfb + kk * 512);
        const uint4 hi = *reinterpret_cast<const uint4*>(ssfb + SFA_BYTES + kk * 512);
        b[8 * kk + 0] = lo.x; b[8 * kk + 1] = lo.y; b[8 * kk + 2] = lo.z; b[8 * kk + 3] = lo.w;
        b[8 * kk + 4] = hi.x; b[8 * kk + 5] = hi.y; b[8 * kk + 6] = hi.z; b[8 * kk + 7] = hi.w;
      }
      __syncwarp();
      const uint32_t sfa_t = tmem + lanes + C::SFA_TMEM0 + slot * SFA_SLOT + q;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) tc_st1(sfa_t + 4 * kk, a[kk]);
      tc_st32(tmem + lanes + C::SFB_TMEM0 + slot * SFB_SLOT, b);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // pairs: on the even CTA's barrier (the odd CTA's stores are complete,
        // waited for above, so a relaxed arrive has nothing left to order)
        if (kPair && rank == 1) mbar_remote_arrive_relaxed(pair_full0 + 8 * slot);
        else mbar_arrive(bar_full + 8 * slot);
      }
    }
    // After an abort the stages this warp did not process still get its
    // arrival, so that the producer's drain of its copies in flight (a wait on
    // the same barriers) completes as soon as they land.
    if (!ok && lane == 0)
      for (int i = 0; i < STAGES && g + i < nstages; ++i) {
        const int slot = (g + i) % STAGES;
        if (kPair && rank == 1) mbar_remote_arrive_relaxed(pair_full0 + 8 * slot);
        else mbar_arrive(bar_full + 8 * slot);
      }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------------------------------------------------------- MMA issuer
    uint32_t stage = 0, phase = 0, aphase = 0;
    bool ok = true, issued = false;
    // Only the weight-tile width changes between tiles, and only when N is not a
    // multiple of 256; otherwise the issuer never decodes a tile (decoding reads
    // global memory, which would leave the tensor pipe idle at tile boundaries).
    // Pairs always have N % 256 == 0.
    const bool uniform_n = kPair || p.N % BN == 0;
    const uint64_t adesc0 = sdesc_kmajor_sw128(sbase);
    const uint64_t bdesc0 = sdesc_kmajor_sw128(sbase + C::OFF_B);
    if (p.test_stall && first_unit < total)
      ok = wait_bounded(bar_never, 0, abort_flag, p.wait_limit_ns, p.status, 6, peer_abort);
    for (int t = first_unit; ok && t < total; t += unit_stride) {
      uint32_t idesc = idesc_nvf4(kPair ? 2 * BM : BM, BN);
      if (!uniform_n) {
        int e, nb, mb, rows, ncols;
        sch.decode(t, 0, e, nb, mb, rows, ncols);
        idesc = idesc_nvf4(BM, ncols);
      }
      // pairs: both CTAs' epilogues arrive on this barrier
      if (!wait_bounded<kPair>(bar_acce, aphase ^ 1, abort_flag, p.wait_limit_ns, p.status, 2, peer_abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < kblocks; ++kb) {
        // pairs: both CTAs' code tiles and scale warps complete this barrier
        if (!wait_bounded<kPair>(bar_full + 8 * stage, phase, abort_flag, p.wait_limit_ns, p.status, 7,
                                 peer_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sfa_t = tmem + C::SFA_TMEM0 + stage * SFA_SLOT;
        const uint32_t sfb_t = tmem + C::SFB_TMEM0 + stage * SFB_SLOT;
        // descriptor start addresses advance by 32 bytes (64 FP4 codes) per k-step
        const uint64_t ad = adesc0 + ((stage * A_BYTES) >> 4);
        const uint64_t bd = bdesc0 + ((stage * C::B_BYTES) >> 4);
        const int nk = kb * 4 + 4 <= ksteps ? 4 : ksteps - kb * 4;
        if (nk == 4) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            if constexpr (kPair)
              tc_mma_nvf4_pair(tmem, ad + 2 * kk, bd + 2 * kk, idesc, sfa_t + 4 * kk, sfb_t + 8 * kk,
                               (kb | kk) != 0 ? 1u : 0u);
            else
              tc_mma_nvf4(tmem, ad + 2 * kk, bd + 2 * kk, idesc, sfa_t + 4 * kk, sfb_t + 8 * kk,
                          (kb | kk) != 0 ? 1u : 0u);
          }
        } else {
          for (int kk = 0; kk < nk; ++kk) {
            if constexpr (kPair)
              tc_mma_nvf4_pair(tmem, ad + 2 * kk, bd + 2 * kk, idesc, sfa_t + 4 * kk, sfb_t + 8 * kk,
                               (kb | kk) != 0 ? 1u : 0u);
            else
              tc_mma_nvf4(tmem, ad + 2 * kk, bd + 2 * kk, idesc, sfa_t + 4 * kk, sfb_t + 8 * kk,
                          (kb | kk) != 0 ? 1u : 0u);
          }
        }
        issued = true;
        // the stage is free in both CTAs once these MMAs are done
        if constexpr (kPair) tc_commit_pair_mc(bar_empty + 8 * stage, 0x3);
        else tc_commit(bar_empty + 8 * stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      if constexpr (kPair) tc_commit_pair_mc(bar_accf, 0x3);
      else tc_commit(bar_accf);
      aphase ^= 1;
    }
    if (!ok && issued) {
      // tensor-core work in flight completes before the tensor memory is freed
      if constexpr (kPair) tc_commit_pair(bar_aux);
      else tc_commit(bar_aux);
      drain_wait(bar_aux, 0);
    }
  } else if (warp >= kFirstEpiWarp && warp < kFirstEpiWarp + kEpiWarps) {
    // ---------------------------------------------------------------- epilogue
    const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
    const int half = (warp - kFirstEpiWarp) >> 2;   // columns [128*half, 128*half + 128)
    const int row = quad * 32 + lane;
    uint32_t aphase = 0;
    const float gs_a = *p.gs_a;
    // The accumulator is released on the barrier the MMA issuer waits on:
    // pairs' odd CTA with one relaxed remote arrive per warp, after every
    // lane's tensor-memory loads were waited for.
    auto release_acc = [&]() {
      if (kPair && rank == 1) {
        __syncwarp();
        if (lane == 0) mbar_remote_arrive_relaxed(pair_acce);
      } else {
        mbar_arrive(bar_acce);
      }
    };
    for (int t = first_unit; t < total; t += unit_stride) {
      int e, nb, mb, rows, ncols;
      sch.decode(t, rank, e, nb, mb, rows, ncols);
      if (!wait_bounded(bar_accf, aphase, abort_flag, p.wait_limit_ns, p.status, 4, peer_abort)) break;
      aphase ^= 1;
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + half * 128;
      const bool active = row < rows && half * 128 < ncols;
      const float alpha = active ? 1.0f / (gs_a * p.gs_b[e]) : 0.0f;
      if constexpr (!kSwiGLU) {
        // BF16 output: each 64-column half is scaled and packed as it leaves
        // TMEM (64 registers instead of 128), then the accumulator is released
        uint32_t packed[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[64];
          tc_ld64_wait(taddr + 64 * c, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(v[2 * i]) * alpha,
                                                     __uint_as_float(v[2 * i + 1]) * alpha);
            packed[32 * c + i] = *reinterpret_cast<uint32_t*>(&b);
          }
        }
        tc_fence_before();
        release_acc();
        if (!active) continue;
        const int64_t orow = (int64_t)p.offsets[e] + mb * BM + row;
        __nv_bfloat16* out = p.c + orow * p.ldc + nb * BN + half * 128;
        // whole 32-byte sectors when the output allows it: a warp's stores go to
        // 32 different rows, and half-sector writes double the store requests
        if (p.c_32B) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_global_32B_stream(out + 16 * j, packed[8 * j], packed[8 * j + 1], packed[8 * j + 2],
                                 packed[8 * j + 3], packed[8 * j + 4], packed[8 * j + 5], packed[8 * j + 6],
                                 packed[8 * j + 7]);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
        }
      } else {
        // columns 32*b + [0,8) gate / [8,16) up of h features 16b..16b+7,
        // columns 32*b + [16,24) gate / [24,32) up of h features 16b+8..16b+15.
        // The first 64 columns become 32 h values before the second 64 are
        // loaded, so at most 96 values are live (the 128-register cap would
        // otherwise spill); the accumulator is released after the second load.
        float hv[32];
        {
          uint32_t u0[64];
          tc_ld64_wait(taddr, u0);
          const float* v0 = reinterpret_cast<const float*>(u0);
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              hv[16 * b + i] = silu(v0[32 * b + i] * alpha) * (v0[32 * b + 8 + i] * alpha);
              hv[16 * b + 8 + i] = silu(v0[32 * b + 16 + i] * alpha) * (v0[32 * b + 24 + i] * alpha);
            }
        }
        uint32_t u1[64];
        tc_ld64_wait(taddr + 64, u1);
        const float* v1 = reinterpret_cast<const float*>(u1);
        tc_fence_before();
        release_acc();
        if (!active) continue;
        const float gs_h = *p.gs_h;
        const int64_t hrow = (int64_t)pad_off[e] + mb * BM + row;
        const int64_t hfeat = (int64_t)nb * (BN / 2) + half * 64;   // first h feature of this thread
        uint32_t words[8];
        uint32_t sfw = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          float h[16];
          if (b < 2) {
#pragma unroll
            for (int i = 0; i < 16; ++i) h[i] = hv[16 * b + i];
          } else {
            const float* v = v1 + 32 * (b - 2);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              h[i] = silu(v[i] * alpha) * (v[8 + i] * alpha);
              h[8 + i] = silu(v[16 + i] * alpha) * (v[24 + i] * alpha);
            }
          }
          const uint32_t sf = quantize_block16(h, gs_h, words[2 * b], words[2 * b + 1]);
          sfw |= sf << (8 * b);
        }
        uint8_t* hc = p.h_codes + hrow * (p.I / 2) + hfeat / 2;   // 32-byte aligned (I % 64 == 0)
        st_global_32B(hc, words[0], words[1], words[2], words[3], words[4], words[5], words[6], words[7]);
        *reinterpret_cast<uint32_t*>(p.h_sf + sf_rows_offset(hrow, hfeat / 16, (p.I + 255) / 256)) = sfw;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) {
    // neither CTA of the pair leaves (or frees its tensor memory) while the
    // other may still arrive on its barriers or run MMAs into its tensor memory
    if (tid == 0) {
      mbar_remote_arrive(mapa_shared(bar_exit, rank ^ 1));
      drain_wait<true>(bar_exit, 0);
    }
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (kPair) tmem_dealloc_pair(tmem, TMEM_COLS);
    else tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Rows of `row_bytes` bytes (K/2 codes), box of 128 bytes x box_rows rows,
// 128-byte swizzle.
bool make_codes_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int g_num_sms = 0;
uint64_t g_wait_limit_ns = 4000000000ull;
int g_test_stall = 0;
int g_gemm_mode = 0;    // 0: one CTA per tile; 1: 2-SM pairs when N % 256 == 0

int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      g_num_sms = n;
  }
  return g_num_sms;
}

template <bool kPair>
size_t smem_bytes(int E) { return (size_t)Cfg<kPair>::OFF_SCHED + 8 * (size_t)(E + 1) + 1024; }

// Clusters of two that can be resident at once for a pair kernel (one CTA per
// SM; a cluster needs two SMs of one GPC), queried once per kernel.
template <bool kSwiGLU>
int pair_clusters(size_t smem) {
  static int cached = -1;
  if (cached < 0) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<true>::OFF_SCHED + 8 * 1025 + 1024;   // the largest request
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel<kSwiGLU, true>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cached = n;
  }
  (void)smem;
  return cached;
}

template <bool kSwiGLU>
int launch_grouped(const uint8_t* a_codes, int64_t a_rows, const uint8_t* b_codes, int N, int K,
                   Params& p, cudaStream_t s) {
  // Pairs need whole 256-column weight tiles (each CTA holds 128 of them).
  const bool pair = g_gemm_mode == 1 && N % BN == 0;
  CUtensorMap ma[4], mb;
  const int boxes[4] = {16, 32, 64, 128};
  for (int i = 0; i < 4; ++i)
    if (!make_codes_map(&ma[i], a_codes, a_rows, K / 2, boxes[i])) return NVFP4MOE_ERR_INVALID;
  if (!make_codes_map(&mb, b_codes, (int64_t)p.E * N, K / 2, pair ? BN / 2 : BN)) return NVFP4MOE_ERR_INVALID;
  int* status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_status) != cudaSuccess)
    return NVFP4MOE_ERR_LAUNCH;
  p.status = status;
  p.wait_limit_ns = g_wait_limit_ns;
  p.test_stall = g_test_stall;
  if (pair) {
    const size_t smem = smem_bytes<true>(p.E);
    auto kern = grouped_gemm_kernel<kSwiGLU, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(Cfg<true>::OFF_SCHED + 8 * 1025 + 1024)) != cudaSuccess)
      return NVFP4MOE_ERR_LAUNCH;
    const int clusters = pair_clusters<kSwiGLU>(smem);
    if (clusters <= 0) return NVFP4MOE_ERR_LAUNCH;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, ma[0], ma[1], ma[2], ma[3], mb, p) != cudaSuccess) return launch_status();
    return launch_status();
  }
  const size_t smem = smem_bytes<false>(p.E);
  auto kern = grouped_gemm_kernel<kSwiGLU, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return NVFP4MOE_ERR_LAUNCH;
  const int grid = num_sms();
  if (grid <= 0) return NVFP4MOE_ERR_LAUNCH;
  kern<<<grid, kThreads, smem, s>>>(ma[0], ma[1], ma[2], ma[3], mb, p);
  return launch_status();
}

int check_common(const uint8_t* a_codes, const uint8_t* a_sf, const float* gs_a, int64_t a_rows,
                 const uint8_t* b_codes, const uint8_t* b_sf, const float* gs_b,
                 const int32_t* offsets, int E, int64_t N, int64_t K) {
  NVFP4_CHECK(E >= 1 && E <= 1024 && K > 0 && K % 64 == 0 && N > 0 && N % 128 == 0,
              NVFP4MOE_ERR_UNSUPPORTED);
  NVFP4_CHECK(K / 2 <= (1ll << 31) && (int64_t)E * N < (1ll << 31) && a_rows < (1ll << 31),
              NVFP4MOE_ERR_UNSUPPORTED);
  NVFP4_CHECK(a_codes && a_sf && gs_a && b_codes && b_sf && gs_b && offsets, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(aligned(a_codes, 16) && aligned(b_codes, 16) && aligned(a_sf, 16) && aligned(b_sf, 16),
              NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(a_rows >= 128 && a_rows % 128 == 0, NVFP4MOE_ERR_INVALID);
  return NVFP4MOE_OK;
}

}  // namespace

int* device_status_word() {
  int* status = nullptr;
  return cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_status) == cudaSuccess ? status : nullptr;
}

uint64_t wait_limit_ns() { return g_wait_limit_ns; }

int device_num_sms() { return num_sms(); }

int test_stall_on() { return g_test_stall; }

}  // namespace nvfp4moe

using namespace nvfp4moe;

extern "C" int nvfp4_grouped_gemm(const uint8_t* a_codes, const uint8_t* a_sf, const float* gs_a,
                                  int64_t a_rows, const uint8_t* b_codes, const uint8_t* b_sf,
                                  const float* gs_b, const int32_t* offsets, int E, int64_t N,
                                  int64_t K, void* c, int64_t ldc, void* stream) {
  NVFP4_TRY(check_common(a_codes, a_sf, gs_a, a_rows, b_codes, b_sf, gs_b, offsets, E, N, K));
  NVFP4_CHECK(c && aligned(c, 16) && ldc >= N && ldc % 8 == 0, NVFP4MOE_ERR_INVALID);
  Params p{};
  p.a_sf = a_sf;
  p.b_sf = b_sf;
  p.gs_a = gs_a;
  p.gs_b = gs_b;
  p.offsets = offsets;
  p.E = E;
  p.N = (int)N;
  p.K = (int)K;
  p.sf_rowtile_bytes = (K / 64) * 512;
  p.a_sf_rowtile_bytes = ((K + 255) / 256) * 2048;
  p.b_sf_expert_bytes = (int64_t)nvfp4_sf_bytes(N, K, NVFP4_SF_TILED);
  p.c = static_cast<__nv_bfloat16*>(c);
  p.ldc = ldc;
  p.c_32B = aligned(c, 32) && ldc % 16 == 0;
  return launch_grouped<false>(a_codes, a_rows, b_codes, (int)N, (int)K, p, as_stream(stream));
}

extern "C" int nvfp4_grouped_gemm_swiglu(const uint8_t* a_codes, const uint8_t* a_sf,
                                         const float* gs_a, int64_t a_rows, const uint8_t* w1_codes,
                                         const uint8_t* w1_sf, const float* gs_w1,
                                         const int32_t* offsets, int E, int64_t I, int64_t K,
                                         const float* gs_h, uint8_t* h_codes, uint8_t* h_sf,
                                         void* stream) {
  NVFP4_CHECK(I > 0 && I % 64 == 0, NVFP4MOE_ERR_UNSUPPORTED);
  NVFP4_TRY(check_common(a_codes, a_sf, gs_a, a_rows, w1_codes, w1_sf, gs_w1, offsets, E, 2 * I, K));
  NVFP4_CHECK(gs_h && h_codes && h_sf && aligned(h_codes, 32) && aligned(h_sf, 16), NVFP4MOE_ERR_INVALID);
  Params p{};
  p.a_sf = a_sf;
  p.b_sf = w1_sf;
  p.gs_a = gs_a;
  p.gs_b = gs_w1;
  p.offsets = offsets;
  p.E = E;
  p.N = (int)(2 * I);
  p.K = (int)K;
  p.sf_rowtile_bytes = (K / 64) * 512;
  p.a_sf_rowtile_bytes = ((K + 255) / 256) * 2048;
  p.b_sf_expert_bytes = (int64_t)nvfp4_sf_bytes(2 * I, K, NVFP4_SF_TILED);
  p.h_codes = h_codes;
  p.h_sf = h_sf;
  p.I = I;
  p.gs_h = gs_h;
  return launch_grouped<true>(a_codes, a_rows, w1_codes, (int)(2 * I), (int)K, p, as_stream(stream));
}

extern "C" int nvfp4moe_last_device_status(void* stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return NVFP4MOE_ERR_LAUNCH;
  int host[2] = {0, 0};
  if (cudaMemcpyFromSymbol(host, g_status, sizeof(host)) != cudaSuccess) return NVFP4MOE_ERR_LAUNCH;
  const int zero[2] = {0, 0};
  if (cudaMemcpyToSymbol(g_status, zero, sizeof(zero)) != cudaSuccess) return NVFP4MOE_ERR_LAUNCH;
  return host[0];
}

extern "C" void nvfp4moe_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns = ns; }

extern "C" void nvfp4moe_set_test_stall(int on) { g_test_stall = on ? 1 : 0; }

extern "C" int nvfp4moe_num_sms(void) { return num_sms(); }

extern "C" int nvfp4moe_set_gemm_mode(int mode) {
  if (mode < 0 || mode > 1) return NVFP4MOE_ERR_INVALID;
  g_gemm_mode = mode;
  return NVFP4MOE_OK;
}
