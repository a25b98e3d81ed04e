// Fused front of the MoE forward ("NVFP4 MegaMoE Kernel" README, "MoE Runner"
// steps 1 and 2; "Bridge Layer": quantize_activation_nvfp4, with a
// pre-computed gs on the CUDA-graph-safe path, else the global scale of x
// computed here): routing, the stable permutation, NVFP4 quantization and the
// scatter into the padded L1 operand, in one cooperative launch.
//
// G blocks; block c owns the contiguous tokens [c*tpb, (c+1)*tpb) and so the
// contiguous flat slots [c*tpb*k, (c+1)*tpb*k).
//   phase 1  route the block's tokens (one warp per token) and histogram
//            their experts -> counts[c][e]; without a pre-computed gs, also
//            max |x| over the block's rows -> one atomicMax
//   -- grid barrier --
//   phase 2  block c turns the columns e = c, c+G, ... into exclusive prefixes
//            over blocks (counts[c'][e] = slots of expert e in blocks < c'),
//            one block-wide scan per column, and writes the column total
//   -- grid barrier --
//   phase 3  every block: exclusive scans of the totals -> offsets (block 0
//            writes them) and padded group starts; the stable position of
//            each of its slots (one warp, 32 slots at a time, grouped with
//            __match_any_sync), then each token row is quantized once and
//            written to the padded rows of its k slots (gs = 2688 / max|x|
//            when it was not given).
// Above NVFP4MOE_FRONT_FUSED_QUANTIZE_MAX_ROWS routed rows the kernel stops
// after the stable positions (block 0 writes the padded group starts) and the
// quantize + scatter runs as a second, full-occupancy kernel (the one of
// moe_quantize_dispatch). Measured on GB300: in the cooperative kernel that
// phase is latency-bound at 2 blocks of 512 threads per SM (64 registers),
// 4.2-4.6 TB/s, against 5.1 TB/s for the separate kernel (one 512-element
// item per warp, 48 warps per SM); the second launch costs ~4 us. Front
// times, quantize inside / as a second kernel: 1024 rows 20 / 24 us, 8192
// rows 27 / 28 us, 32768 rows 63 / 64 us, 65536 rows 138 / 122 us, 131072
// rows 270 / 224 us.
// The same permutation as moe_permute (a stable counting sort by expert of
// the flat slots t*k + j), the same rows as moe_quantize_dispatch.
//
// The grid barriers are bounded: one that does not complete within the wait
// limit sets the device status to NVFP4MOE_ERR_DEVICE_TIMEOUT (wait site 8 or
// 9) and the kernel returns. Offsets, flat_to_perm (and the padded group
// starts when a second kernel quantizes) are zeroed before the first barrier,
// so the later stages then find no rows and read nothing out of bounds.
#include "common.cuh"

namespace nvfp4moe {

// Quantize + scatter of moe_quantize_dispatch (defined in quantize.cu), given
// the padded group starts pad_off[e] (e < E) and either gs_in or the bits of
// max|x| (the global scale is then 2688 / max|x|, written to gs_out when that
// is not null).
int launch_dispatch_quantize(const void* x, int64_t T, int64_t K, int64_t ldx, int k, const float* gs_in,
                             const uint32_t* amax_bits, float* gs_out, const int32_t* topk_ids,
                             const int32_t* offsets, const int32_t* flat_to_perm, const int32_t* pad_off,
                             uint8_t* a_codes, uint8_t* a_sf, cudaStream_t s);

namespace {

constexpr int kFrontThreads = 512;
constexpr int kFrontMaxSlots = 4096;   // flat slots per block (tpb * k)
constexpr int kFrontMaxBlocks = 1024;

struct FrontParams {
  const __nv_bfloat16* x;
  int64_t ldx;
  const float* logits;
  int64_t T;
  int K, E, k, tpb;
  const float* gs_x;       // pre-computed global scale, or null: computed from max|x|
  float* gs_out;           // null, or receives the global scale used
  uint32_t* amax_bits;     // max|x| as f32 bits (zeroed before the launch)
  int32_t* ids;
  float* w;
  int32_t* offsets;
  int32_t* p2f;
  int32_t* f2p;
  uint8_t* a_codes;
  uint8_t* a_sf;
  int32_t* counts;        // [G][E]
  int32_t* totals;        // [E]
  int32_t* pad_out;       // [E] padded group starts, written when !quantize
  int quantize;           // 1: quantize + scatter here; 0: stop after the positions
  unsigned int* barrier;  // zeroed before the launch
  uint64_t limit_ns;
  int* status;
  int test_stall;         // block 0 leaves before the first grid barrier
};

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// All blocks of the (cooperative) grid arrive; false if the wait timed out.
__device__ bool grid_barrier(const FrontParams& p, unsigned int target, int site, int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(p.barrier, 1u);
    int ok = 1;
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire_gpu(p.barrier) < target) {
      if (global_timer_ns() - t0 > p.limit_ns) {
        ok = 0;
        if (atomicCAS(&p.status[0], 0, NVFP4MOE_ERR_DEVICE_TIMEOUT) == 0) p.status[1] = site;
        break;
      }
    }
    *flag = ok;
  }
  __syncthreads();
  return *flag != 0;
}

// Block-wide exclusive scan of n <= 2 * kFrontThreads values in place (smem).
__device__ void block_exclusive_scan(int32_t* a, int n, int32_t* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = 2 * tid, i1 = 2 * tid + 1;
  const int v0 = i0 < n ? a[i0] : 0, v1 = i1 < n ? a[i1] : 0;
  const int pair = v0 + v1;
  int incl = pair;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int s = lane < kFrontThreads / 32 ? warp_tot[lane] : 0;
    int si = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, si, d);
      if (lane >= d) si += y;
    }
    if (lane < kFrontThreads / 32) warp_tot[lane] = si - s;
  }
  __syncthreads();
  const int excl = warp_tot[warp] + incl - pair;
  if (i0 < n) a[i0] = excl;
  if (i1 < n) a[i1] = excl + v0;
  __syncthreads();
}

template <int VPL>
__global__ void __launch_bounds__(kFrontThreads) moe_front_kernel(const FrontParams p) {
  extern __shared__ int32_t sm[];
  const int E = p.E, k = p.k;
  int32_t* next = sm;                    // [E]
  int32_t* offs = next + E;              // [E + 1]
  int32_t* pad = offs + (E + 1);         // [E + 1]
  int32_t* slot_e = pad + (E + 1);       // [tpb * k]
  int32_t* slot_pos = slot_e + p.tpb * k;
  int32_t* misc = slot_pos + p.tpb * k;  // [32]: warp totals, barrier flag
  int32_t* col = misc + 32;              // [G]: one expert's counts over the blocks
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = kFrontThreads / 32;
  const int G = gridDim.x, c = blockIdx.x;
  const int64_t t0 = (int64_t)c * p.tpb;
  const int64_t t1 = t0 + p.tpb < p.T ? t0 + p.tpb : p.T;
  const int ntok = t1 > t0 ? (int)(t1 - t0) : 0;
  const int nslot = ntok * k;

  // ---- phase 1: route, histogram; safe offsets / flat_to_perm first
  for (int e = tid; e < E; e += kFrontThreads) next[e] = 0;
  if (c == 0) {
    for (int e = tid; e <= E; e += kFrontThreads) p.offsets[e] = 0;
    if (!p.quantize)   // read by the quantize kernel that follows, even after a timeout
      for (int e = tid; e < E; e += kFrontThreads) p.pad_out[e] = 0;
  }
  for (int s = tid; s < nslot; s += kFrontThreads) p.f2p[t0 * k + s] = 0;
  __syncthreads();
  for (int tl = warp; tl < ntok; tl += nwarps) {
    const int64_t t = t0 + tl;
    int my_i;
    float my_w;
    route_token<VPL>(p.logits + t * E, E, k, lane, my_i, my_w);
    if (lane < k) {
      p.ids[t * k + lane] = my_i;
      p.w[t * k + lane] = my_w;
      slot_e[tl * k + lane] = my_i;
      atomicAdd(&next[my_i], 1);
    }
  }
  if (!p.gs_x) {
    // max |x| over the block's rows, four 16-byte loads in flight per thread
    const int vpr = p.K / 8;
    const int nvec = ntok * vpr;
    float m = 0.0f;
    for (int i0 = tid; i0 < nvec; i0 += 4 * kFrontThreads) {
      uint4 u[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j * kFrontThreads;
        u[j] = make_uint4(0u, 0u, 0u, 0u);
        if (i < nvec) {
          const int tl = i / vpr;
          u[j] = __ldg(reinterpret_cast<const uint4*>(p.x + (t0 + tl) * p.ldx) + (i - tl * vpr));
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float f[8];
        bf16x8_to_f32(u[j], f);
#pragma unroll
        for (int q = 0; q < 8; ++q) m = fmaxf(m, fabsf(f[q]));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) misc[warp] = (int32_t)__float_as_uint(m);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kFrontThreads) p.counts[(int64_t)c * E + e] = next[e];
  if (!p.gs_x && tid == 0) {
    uint32_t mb = 0;
    for (int i = 0; i < nwarps; ++i) mb = max(mb, (uint32_t)misc[i]);   // non-negative f32 bits order as floats
    if (mb > 0) atomicMax(p.amax_bits, mb);
  }
  if (p.test_stall && c == 0) return;
  if (!grid_barrier(p, (unsigned)G, 8, misc + 31)) return;

  // ---- phase 2: per expert column, exclusive prefix over blocks and total
  for (int e = c; e < E; e += G) {
    for (int cc = tid; cc < G; cc += kFrontThreads) col[cc] = __ldcg(p.counts + (int64_t)cc * E + e);
    __syncthreads();
    const int last = tid == 0 ? col[G - 1] : 0;     // the scan reads before it writes
    block_exclusive_scan(col, G, misc);
    for (int cc = tid; cc < G; cc += kFrontThreads) p.counts[(int64_t)cc * E + e] = col[cc];
    if (tid == 0) p.totals[e] = col[G - 1] + last;
    __syncthreads();
  }
  if (!grid_barrier(p, 2u * G, 9, misc + 31)) return;

  // ---- phase 3: offsets, padded starts, stable positions, quantize + scatter
  for (int e = tid; e < E; e += kFrontThreads) {
    const int n = __ldcg(p.totals + e);
    offs[e] = n;
    pad[e] = (n + 127) / 128 * 128;
  }
  __syncthreads();
  block_exclusive_scan(offs, E, misc);
  block_exclusive_scan(pad, E, misc);
  if (c == 0) {
    for (int e = tid; e < E; e += kFrontThreads) p.offsets[e] = offs[e];
    if (tid == 0) p.offsets[E] = (int32_t)(p.T * k);
  }
  for (int e = tid; e < E; e += kFrontThreads) next[e] = offs[e] + __ldcg(p.counts + (int64_t)c * E + e);
  __syncthreads();
  if (warp == 0) {
    for (int i = 0; i < nslot; i += 32) {
      const int s = i + lane;
      const bool valid = s < nslot;
      const int e = valid ? slot_e[s] : -1 - lane;  // invalid lanes never match a real expert
      const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int start = valid ? next[e] : 0;
      __syncwarp();
      if (valid) {
        const int pos = start + rank;
        const int64_t f = t0 * k + s;
        slot_pos[s] = pos;
        p.p2f[pos] = (int32_t)f;
        p.f2p[f] = pos;
        if (lane == 31 - __clz(peers)) next[e] = start + __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (!p.quantize) {
    if (c == 0)
      for (int e = tid; e < E; e += kFrontThreads) p.pad_out[e] = pad[e];
    return;
  }
  const float gs = p.gs_x ? *p.gs_x : global_scale_from_amax_bits(__ldcg(p.amax_bits));
  if (p.gs_out && c == 0 && tid == 0) *p.gs_out = gs;
  const int nchunk = (p.K + 511) / 512;
  const int64_t s_tiles = (p.K + 255) / 256;
  // item = (token, 512-element chunk); each warp loads its next item's 32
  // bytes per lane while it quantizes and scatters the current one (measured
  // at prefill: 0.136 against 0.143 ms)
  const int nitem = ntok * nchunk;
  auto load_item = [&](int item, uint4 (&r)[2]) {
    const int tl = item / nchunk;
    const int64_t col0 = (int64_t)(item - tl * nchunk) * 512 + lane * 16;
    if (item < nitem && col0 < p.K) {
      const uint4* src = reinterpret_cast<const uint4*>(p.x + (t0 + tl) * p.ldx + col0);
      r[0] = __ldg(src);
      r[1] = __ldg(src + 1);
    } else {
      r[0] = r[1] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  uint4 cur[2], nxt[2];
  load_item(warp, cur);
  for (int item = warp; item < nitem; item += nwarps) {
    load_item(item + nwarps, nxt);
    const int tl = item / nchunk;
    const int64_t col0 = (int64_t)(item - tl * nchunk) * 512 + lane * 16;
    const bool valid = col0 < p.K;
    // lane j < k: the padded row of the token's slot j, as the row parts of
    // its code and scale addresses
    unsigned long long my_codes = 0, my_sf = 0;
    if (lane < k) {
      const int e = slot_e[tl * k + lane];
      const int64_t prow = (int64_t)pad[e] + slot_pos[tl * k + lane] - offs[e];
      my_codes = reinterpret_cast<unsigned long long>(p.a_codes + prow * (p.K / 2));
      my_sf = reinterpret_cast<unsigned long long>(p.a_sf + sf_rows_row_part(prow, s_tiles));
    }
    float v[16];
    bf16x8_to_f32(cur[0], v);
    bf16x8_to_f32(cur[1], v + 8);
    uint32_t w0 = 0, w1 = 0;
    const uint32_t s = quantize_block16(v, gs, w0, w1);   // zeros past K: scale 0
    cur[0] = nxt[0];
    cur[1] = nxt[1];
    const uint32_t word = gather_sf_word(s);
    const int64_t code_col = col0 / 2, sf_col = sf_rows_block_part(col0 / 16);
    for (int j = 0; j < k; ++j) {
      uint8_t* dc = reinterpret_cast<uint8_t*>(__shfl_sync(0xFFFFFFFFu, my_codes, j));
      uint8_t* ds = reinterpret_cast<uint8_t*>(__shfl_sync(0xFFFFFFFFu, my_sf, j));
      if (valid) st_global_8B_stream(dc + code_col, w0, w1);
      if (valid && (lane & 3) == 0) *reinterpret_cast<uint32_t*>(ds + sf_col) = word;
    }
  }
}

size_t front_smem_bytes(int E, int slots) { return (size_t)(3 * E + 2 + 2 * slots + 32 + kFrontMaxBlocks) * 4; }

template <int VPL>
int launch_front_vpl(FrontParams& p, int G, size_t smem, cudaStream_t s) {
  auto kern = moe_front_kernel<VPL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return NVFP4MOE_ERR_LAUNCH;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(kFrontThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return NVFP4MOE_ERR_LAUNCH;
  return launch_status();
}

template <int VPL>
int max_coresident(size_t smem) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, moe_front_kernel<VPL>, kFrontThreads, smem) !=
      cudaSuccess)
    return 0;
  return per_sm * device_num_sms();
}

int vpl_of(int E) { return E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : E <= 512 ? 16 : 32; }

}  // namespace

size_t front_workspace_bytes(int64_t T, int E) {
  const int64_t g = T < kFrontMaxBlocks ? T : kFrontMaxBlocks;
  return 256 + 2 * (size_t)ceil_div((int64_t)E * 4, 256) * 256 + (size_t)ceil_div(g * E * 4, 256) * 256;
}

bool moe_front_fits(int64_t T, int E, int k) {
  if (T < 1 || k < 1 || k > 16 || k > E || E > 1024) return false;
  const size_t smem_max = front_smem_bytes(E, kFrontMaxSlots);
  const int vpl = vpl_of(E);
  int gmax = vpl == 1 ? max_coresident<1>(smem_max) : vpl == 2 ? max_coresident<2>(smem_max)
           : vpl == 4 ? max_coresident<4>(smem_max) : vpl == 8 ? max_coresident<8>(smem_max)
           : vpl == 16 ? max_coresident<16>(smem_max) : max_coresident<32>(smem_max);
  if (gmax > kFrontMaxBlocks) gmax = kFrontMaxBlocks;
  if (gmax < 1) return false;
  const int64_t G = T < gmax ? T : gmax;
  return ceil_div(T, G) * k <= kFrontMaxSlots;
}

int moe_front(const void* x, int64_t ldx, const float* logits, int64_t T, int64_t K, int E, int k,
              const float* gs_x, float* gs_out, int32_t* ids, float* w, int32_t* offsets, int32_t* p2f,
              int32_t* f2p, uint8_t* a_codes, uint8_t* a_sf, void* ws, size_t ws_bytes, cudaStream_t s) {
  NVFP4_CHECK(T >= 1 && K % 64 == 0 && k >= 1 && k <= 16 && k <= E && E <= 1024, NVFP4MOE_ERR_UNSUPPORTED);
  NVFP4_CHECK(ws && ws_bytes >= front_workspace_bytes(T, E) && aligned(ws, 256), NVFP4MOE_ERR_WORKSPACE);
  const size_t smem_max = front_smem_bytes(E, kFrontMaxSlots);
  const int vpl = vpl_of(E);
  int gmax = vpl == 1 ? max_coresident<1>(smem_max) : vpl == 2 ? max_coresident<2>(smem_max)
           : vpl == 4 ? max_coresident<4>(smem_max) : vpl == 8 ? max_coresident<8>(smem_max)
           : vpl == 16 ? max_coresident<16>(smem_max) : max_coresident<32>(smem_max);
  if (gmax > kFrontMaxBlocks) gmax = kFrontMaxBlocks;
  NVFP4_CHECK(gmax >= 1, NVFP4MOE_ERR_LAUNCH);
  int G = (int)(T < gmax ? T : gmax);
  const int tpb = (int)ceil_div(T, G);
  G = (int)ceil_div(T, tpb);
  NVFP4_CHECK((int64_t)tpb * k <= kFrontMaxSlots, NVFP4MOE_ERR_UNSUPPORTED);
  FrontParams p{};
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.ldx = ldx;
  p.logits = logits;
  p.T = T;
  p.K = (int)K;
  p.E = E;
  p.k = k;
  p.tpb = tpb;
  p.gs_x = gs_x;
  p.gs_out = gs_out;
  p.ids = ids;
  p.w = w;
  p.offsets = offsets;
  p.p2f = p2f;
  p.f2p = f2p;
  p.a_codes = a_codes;
  p.a_sf = a_sf;
  uint8_t* wb = static_cast<uint8_t*>(ws);
  p.barrier = reinterpret_cast<unsigned int*>(wb);
  p.amax_bits = reinterpret_cast<uint32_t*>(wb + 4);
  const int64_t e_bytes = ceil_div((int64_t)E * 4, 256) * 256;
  p.totals = reinterpret_cast<int32_t*>(wb + 256);
  p.pad_out = reinterpret_cast<int32_t*>(wb + 256 + e_bytes);
  p.counts = reinterpret_cast<int32_t*>(wb + 256 + 2 * e_bytes);
  p.quantize = T * k <= NVFP4MOE_FRONT_FUSED_QUANTIZE_MAX_ROWS ? 1 : 0;
  p.limit_ns = wait_limit_ns();
  p.status = device_status_word();
  p.test_stall = test_stall_on();
  NVFP4_CHECK(p.status, NVFP4MOE_ERR_LAUNCH);
  if (cudaMemsetAsync(p.barrier, 0, 2 * sizeof(unsigned int), s) != cudaSuccess) return NVFP4MOE_ERR_LAUNCH;
  const size_t smem = front_smem_bytes(E, tpb * k);
  int st;
  switch (vpl) {
    case 1: st = launch_front_vpl<1>(p, G, smem, s); break;
    case 2: st = launch_front_vpl<2>(p, G, smem, s); break;
    case 4: st = launch_front_vpl<4>(p, G, smem, s); break;
    case 8: st = launch_front_vpl<8>(p, G, smem, s); break;
    case 16: st = launch_front_vpl<16>(p, G, smem, s); break;
    default: st = launch_front_vpl<32>(p, G, smem, s); break;
  }
  if (st != NVFP4MOE_OK || p.quantize) return st;
  // After a barrier timeout the cooperative kernel leaves offsets,
  // flat_to_perm and the padded starts zeroed, so this kernel writes every
  // slot into padded row 0: only inside the padded operand.
  return launch_dispatch_quantize(x, T, K, ldx, k, gs_x, gs_x ? nullptr : p.amax_bits, gs_out, ids, offsets,
                                  f2p, p.pad_out, a_codes, a_sf, s);
}

}  // namespace nvfp4moe
