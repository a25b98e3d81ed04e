// BF16 -> NVFP4 quantization kernels ("NVFP4 MegaMoE Kernel" README,
// "Bridge Layer": quantize_to_nvfp4 / quantize_activation_nvfp4, and
// "Correctness Bugs Fixed" bugs 3 and 4 for the zero and underflow blocks).
//
// Work split: one warp quantizes 512 consecutive elements of one row, one
// 16-element block per lane: each lane reads 32 contiguous bytes, the warp
// 1 KB (coalesced), writes 8 code bytes per lane (256 contiguous bytes) and
// the 32 scale bytes as eight 4-byte words of the tiled scale layout.
#include "common.cuh"

namespace nvfp4moe {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kChunk = 512;  // elements per warp

// Largest |x| over the rows read, as the bit pattern of a non-negative f32
// (atomicMax on the bits orders non-negative floats correctly). Each thread
// keeps four 16-byte loads in flight; kContig: no row gather and ldx == cols,
// so the rows are one flat array.
template <bool kContig>
__global__ void __launch_bounds__(256) amax_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                        int64_t rows, int64_t cols, int64_t ldx,
                                                        const int32_t* __restrict__ row_src,
                                                        uint32_t* __restrict__ amax_bits) {
  const int64_t vec_per_row = cols / 8;
  const int64_t total = rows * vec_per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  float m = 0.0f;
  for (int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i0 < total; i0 += 4 * stride) {
    uint4 u[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t i = i0 + j * stride;
      u[j] = make_uint4(0u, 0u, 0u, 0u);
      if (i < total) {
        if (kContig) {
          u[j] = __ldg(reinterpret_cast<const uint4*>(x) + i);
        } else {
          const int64_t r = i / vec_per_row, v = i - r * vec_per_row;
          const int64_t src = row_src ? row_src[r] : r;
          if (src >= 0) u[j] = __ldg(reinterpret_cast<const uint4*>(x + src * ldx) + v);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float f[8];
      bf16x8_to_f32(u[j], f);
#pragma unroll
      for (int c = 0; c < 8; ++c) m = fmaxf(m, fabsf(f[c]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0 && m > 0.0f) atomicMax(amax_bits, __float_as_uint(m));
}

__device__ __forceinline__ float load_gs(const float* gs_in, const uint32_t* amax_bits) {
  return gs_in ? *gs_in : global_scale_from_amax_bits(*amax_bits);
}

__global__ void __launch_bounds__(256) quantize_rows_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
    const float* gs_in, const uint32_t* amax_bits, float* gs_out,
    const int32_t* __restrict__ row_src, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
    int sf_layout) {
  const float gs = load_gs(gs_in, amax_bits);
  if (gs_out && blockIdx.x == 0 && threadIdx.x == 0) *gs_out = gs;
  const int lane = threadIdx.x & 31;
  const int64_t nchunk = (cols + kChunk - 1) / kChunk;
  const int64_t gw = blockIdx.x * (int64_t)kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t r = gw / nchunk;
  if (r >= rows) return;
  const int64_t col0 = (gw - r * nchunk) * kChunk + lane * 16;
  const bool valid = col0 < cols;
  const int64_t src = row_src ? (int64_t)row_src[r] : r;
  uint32_t w0 = 0, w1 = 0, s = 0;
  if (valid) s = quantize_lane16(src >= 0 ? x + src * ldx : nullptr, col0, gs, w0, w1);
  if (valid) *reinterpret_cast<uint2*>(codes + r * (cols / 2) + col0 / 2) = make_uint2(w0, w1);
  if (sf_layout == NVFP4_SF_TILED) {
    const uint32_t word = gather_sf_word(s);
    if (valid && (lane & 3) == 0)
      *reinterpret_cast<uint32_t*>(sf + sf_tiled_offset(r, col0 / 16, (cols + 63) / 64)) = word;
  } else if (sf_layout == NVFP4_SF_TILED_ROWS) {
    const uint32_t word = gather_sf_word(s);
    if (valid && (lane & 3) == 0)
      *reinterpret_cast<uint32_t*>(sf + sf_rows_offset(r, col0 / 16, (cols + 255) / 256)) = word;
  } else if (valid) {
    sf[r * (cols / 16) + col0 / 16] = static_cast<uint8_t>(s);
  }
}

// Padded group starts P_e = 128 * sum_{e'<e} ceil(n_e'/128), one warp.
__global__ void padded_offsets_kernel(const int32_t* __restrict__ offsets, int E,
                                      int32_t* __restrict__ pad_off) {
  const int lane = threadIdx.x;
  int carry = 0;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    const int mt = e < E ? (offsets[e + 1] - offsets[e] + 127) >> 7 : 0;
    int incl = mt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += y;
    }
    if (e < E) pad_off[e] = (carry + incl - mt) * 128;
    carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  if (lane == 0) pad_off[E] = carry * 128;
}

// Each token row is quantized once and written to the padded row of each of
// its k routed slots.
__global__ void __launch_bounds__(256) dispatch_quantize_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t T, int64_t K, int64_t ldx, int k,
    const float* gs_in, const uint32_t* amax_bits, float* gs_out,
    const int32_t* __restrict__ topk_ids, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ flat_to_perm, const int32_t* __restrict__ pad_off,
    uint8_t* __restrict__ a_codes, uint8_t* __restrict__ a_sf) {
  const float gs = load_gs(gs_in, amax_bits);
  if (gs_out && blockIdx.x == 0 && threadIdx.x == 0) *gs_out = gs;
  const int lane = threadIdx.x & 31;
  const int64_t nchunk = (K + kChunk - 1) / kChunk;
  const int64_t gw = blockIdx.x * (int64_t)kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t t = gw / nchunk;
  if (t >= T) return;
  const int64_t col0 = (gw - t * nchunk) * kChunk + lane * 16;
  const bool valid = col0 < K;
  // lane j < k finds the padded row of slot j while the row is being quantized,
  // and the row parts of its code and scale addresses (the warp's lanes then
  // only add their column parts)
  const int64_t s_tiles = (K + 255) / 256;
  unsigned long long my_codes = 0, my_sf = 0;
  if (lane < k) {
    const int64_t f = t * k + lane;
    const int e = topk_ids[f];
    const int64_t prow = pad_off[e] + flat_to_perm[f] - offsets[e];
    my_codes = reinterpret_cast<unsigned long long>(a_codes + prow * (K / 2));
    my_sf = reinterpret_cast<unsigned long long>(a_sf + sf_rows_row_part(prow, s_tiles));
  }
  uint32_t w0 = 0, w1 = 0, s = 0;
  if (valid) s = quantize_lane16(x + t * ldx, col0, gs, w0, w1);
  const uint32_t word = gather_sf_word(s);
  const int64_t code_col = col0 / 2, sf_col = sf_rows_block_part(col0 / 16);
  for (int j = 0; j < k; ++j) {
    uint8_t* dc = reinterpret_cast<uint8_t*>(__shfl_sync(0xFFFFFFFFu, my_codes, j));
    uint8_t* ds = reinterpret_cast<uint8_t*>(__shfl_sync(0xFFFFFFFFu, my_sf, j));
    // codes stream past L2 (264 MB at 65536 rows); the scale words, four bytes
    // of a 32-byte sector from each of eight rows, stay until their sector is whole
    if (valid) st_global_8B_stream(dc + code_col, w0, w1);
    if (valid && (lane & 3) == 0) *reinterpret_cast<uint32_t*>(ds + sf_col) = word;
  }
}

// RMS norm -> RoPE -> NVFP4 quantization (README "THE PLAN", item 3: "Q norm
// -> RoPE -> NVFP4 quant" in one pass).
//
// A row of nb = D/16 blocks is handled by a group of G lanes (G a power of two,
// 4 <= G <= 32) whose lanes own up to BPL = 3 blocks each (lane l: blocks l,
// l + G, ...), held in registers as BF16, so the row is read once; each group
// strides over rows. Measured on the 192-wide q-head rows: keeping only the
// BF16 words live (each block is widened to f32 twice, for the sum of squares
// and for the rest) lets 3 blocks of 256 threads share an SM, 25% faster than
// 2 blocks that also held the f32 values and the next row's loads. Rows of
// more than 96 blocks take the second kernel below, which streams the row
// twice. Per row: the sum of squares (per lane in
// block order, then a butterfly over the group), y = x * (1/sqrt(mean + eps))
// * gamma, the adjacent pairs of the rope blocks rotated with the tables at
// the row's position, then each block quantized with the pre-computed global
// scale. Scale bytes of 4 consecutive blocks are gathered into one 4-byte
// store. A position outside [0, max_pos) zeroes the row's output and records
// NVFP4MOE_ERR_INVALID in the device status word.
struct NormRopeArgs {
  const __nv_bfloat16* x;
  int64_t rows, D, ldx;
  const float* gamma;
  float eps;
  int64_t R;
  const int32_t* positions;
  const float* cos_t;
  const float* sin_t;
  int64_t max_pos;
  const float* gs;
  uint8_t* codes;
  uint8_t* sf;
  int sf_layout;
  float* y_out;
  int* status;
};

__device__ __forceinline__ void norm_rope_block(const NormRopeArgs& a, int64_t b, int64_t rope0, int32_t pos,
                                                bool bad, float inv, float (&v)[16]) {
  float g[16];
  const float4* gp = reinterpret_cast<const float4*>(a.gamma + 16 * b);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 t = __ldg(gp + i);
    g[4 * i] = t.x; g[4 * i + 1] = t.y; g[4 * i + 2] = t.z; g[4 * i + 3] = t.w;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = v[i] * inv * g[i];
  if (b >= rope0 && !bad) {
    const int64_t half = a.R / 2, j0 = (b - rope0) * 8;
    const float4* ct = reinterpret_cast<const float4*>(a.cos_t + (int64_t)pos * half + j0);
    const float4* st = reinterpret_cast<const float4*>(a.sin_t + (int64_t)pos * half + j0);
    const float4 c0 = __ldg(ct), c1 = __ldg(ct + 1), s0 = __ldg(st), s1 = __ldg(st + 1);
    const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float c = cs[j], s = sn[j];
      const float x0 = v[2 * j], x1 = v[2 * j + 1];
      v[2 * j] = x0 * c - x1 * s;
      v[2 * j + 1] = x0 * s + x1 * c;
    }
  }
  if (bad) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
  }
}

// Quantize block b of row r and store codes, y; returns the scale byte.
__device__ __forceinline__ uint32_t norm_rope_store(const NormRopeArgs& a, int64_t r, int64_t b, float gs,
                                                    const float (&v)[16]) {
  uint32_t w0, w1;
  const uint32_t sfb = quantize_block16(v, gs, w0, w1);
  *reinterpret_cast<uint2*>(a.codes + r * (a.D / 2) + 8 * b) = make_uint2(w0, w1);
  if (a.y_out) {
    float4* yo = reinterpret_cast<float4*>(a.y_out + r * a.D + 16 * b);
#pragma unroll
    for (int i = 0; i < 4; ++i) yo[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
  return sfb;
}

// Scale byte of block b of row r; `word` holds the bytes of blocks b..b+3 in
// the lane whose block is a multiple of 4 (words only when the 4 bytes are
// contiguous and aligned in the layout).
__device__ __forceinline__ void norm_rope_store_sf(const NormRopeArgs& a, int64_t r, int64_t b, uint32_t sfb,
                                                   uint32_t word, bool words) {
  const int64_t nb = a.D / 16;
  auto offset = [&](int64_t bb) {
    return a.sf_layout == NVFP4_SF_TILED        ? sf_tiled_offset(r, bb, (a.D + 63) / 64)
           : a.sf_layout == NVFP4_SF_TILED_ROWS ? sf_rows_offset(r, bb, (a.D + 255) / 256)
                                                : r * nb + bb;
  };
  if (words) {
    if ((b & 3) == 0) *reinterpret_cast<uint32_t*>(a.sf + offset(b)) = word;
  } else {
    a.sf[offset(b)] = static_cast<uint8_t>(sfb);
  }
}

template <int G, int BPL>
__global__ void __launch_bounds__(256, 3) norm_rope_quantize_kernel(const NormRopeArgs a) {
  const int lane = threadIdx.x & 31, gl = lane % G;
  const unsigned gmask = G == 32 ? 0xFFFFFFFFu : (((1u << G) - 1u) << (lane - gl));
  const int64_t ngroups = (int64_t)gridDim.x * blockDim.x / G;
  const int64_t nb = a.D / 16, rope0 = (a.D - a.R) / 16;
  const float gs = *a.gs;
  // 4-byte scale words need 4 consecutive blocks in 4 consecutive lanes
  const bool words = (nb % 4) == 0 && G >= 4;
  auto load_row = [&](int64_t r, uint4 (&raw)[BPL][2]) {
    const __nv_bfloat16* xr = a.x + r * a.ldx;
#pragma unroll
    for (int i = 0; i < BPL; ++i) {
      const int64_t b = gl + (int64_t)G * i;
      if (b < nb) {
        const uint4* p = reinterpret_cast<const uint4*>(xr + 16 * b);
        raw[i][0] = __ldg(p);
        raw[i][1] = __ldg(p + 1);
      }
    }
  };
  int64_t r = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / G;
  uint4 cur[BPL][2];
  for (; r < a.rows; r += ngroups) {     // group-uniform: whole groups loop together
    load_row(r, cur);
    const int32_t pos = a.R > 0 ? a.positions[r] : 0;
    const bool bad = a.R > 0 && (pos < 0 || pos >= a.max_pos);
    if (bad && gl == 0 && atomicCAS(&a.status[0], 0, NVFP4MOE_ERR_INVALID) == 0) a.status[1] = 10;
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < BPL; ++i) {
      const int64_t b = gl + (int64_t)G * i;
      if (b < nb) {
        float v[16];
        bf16x8_to_f32(cur[i][0], v);
        bf16x8_to_f32(cur[i][1], v + 8);
#pragma unroll
        for (int e = 0; e < 16; ++e) ss = fmaf(v[e], v[e], ss);
      }
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(gmask, ss, o);
    const float inv = rsqrtf(ss / (float)a.D + a.eps);
#pragma unroll
    for (int i = 0; i < BPL; ++i) {
      const int64_t b = gl + (int64_t)G * i;
      uint32_t sfb = 0;
      if (b < nb) {
        float v[16];
        bf16x8_to_f32(cur[i][0], v);
        bf16x8_to_f32(cur[i][1], v + 8);
        norm_rope_block(a, b, rope0, pos, bad, inv, v);
        sfb = norm_rope_store(a, r, b, gs, v);
      }
      const uint32_t b1 = __shfl_down_sync(gmask, sfb, 1, G);
      const uint32_t b2 = __shfl_down_sync(gmask, sfb, 2, G);
      const uint32_t b3 = __shfl_down_sync(gmask, sfb, 3, G);
      if (b < nb) norm_rope_store_sf(a, r, b, sfb, sfb | (b1 << 8) | (b2 << 16) | (b3 << 24), words);
    }
  }
}

// Long rows: one warp per row, the row streamed twice (sum of squares, then
// the rest); scale bytes stored one by one.
__global__ void __launch_bounds__(256) norm_rope_quantize_long_kernel(const NormRopeArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= a.rows) return;
  const int64_t nb = a.D / 16, rope0 = (a.D - a.R) / 16;
  const __nv_bfloat16* xr = a.x + r * a.ldx;
  const int32_t pos = a.R > 0 ? a.positions[r] : 0;
  const bool bad = a.R > 0 && (pos < 0 || pos >= a.max_pos);
  if (bad && lane == 0 && atomicCAS(&a.status[0], 0, NVFP4MOE_ERR_INVALID) == 0) a.status[1] = 10;
  float ss = 0.0f;
  for (int64_t b = lane; b < nb; b += 32) {
    float v[16];
    const uint4* p = reinterpret_cast<const uint4*>(xr + 16 * b);
    bf16x8_to_f32(__ldg(p), v);
    bf16x8_to_f32(__ldg(p + 1), v + 8);
#pragma unroll
    for (int i = 0; i < 16; ++i) ss = fmaf(v[i], v[i], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  const float inv = rsqrtf(ss / (float)a.D + a.eps);
  const float gs = *a.gs;
  for (int64_t b = lane; b < nb; b += 32) {
    float v[16];
    const uint4* p = reinterpret_cast<const uint4*>(xr + 16 * b);
    bf16x8_to_f32(__ldg(p), v);
    bf16x8_to_f32(__ldg(p + 1), v + 8);
    norm_rope_block(a, b, rope0, pos, bad, inv, v);
    const uint32_t sfb = norm_rope_store(a, r, b, gs, v);
    norm_rope_store_sf(a, r, b, sfb, 0u, false);
  }
}

template <int G, int BPL>
void launch_norm_rope(const NormRopeArgs& a, cudaStream_t s) {
  // as many blocks as are resident at once (each strides over the rows), no
  // more than the rows need
  static int per_sm = 0;
  if (per_sm == 0 &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, norm_rope_quantize_kernel<G, BPL>, 256, 0) != cudaSuccess)
    per_sm = 0;
  const int64_t groups_per_block = 256 / G;
  const int64_t want = (int64_t)device_num_sms() * (per_sm > 0 ? per_sm : 2);
  const int64_t need = ceil_div(a.rows, groups_per_block);
  norm_rope_quantize_kernel<G, BPL><<<(unsigned)(need < want ? need : want), 256, 0, s>>>(a);
}

int launch_amax(const void* x, int64_t rows, int64_t cols, int64_t ldx, const int32_t* row_src,
                uint32_t* amax_bits, cudaStream_t s) {
  if (cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), s) != cudaSuccess) return NVFP4MOE_ERR_LAUNCH;
  const int64_t total = rows * (cols / 8);
  if (total > 0) {
    // 8 blocks of 256 threads per SM, fewer when there is not enough work for
    // four loads per thread
    const int64_t blocks = ceil_div(total, 256 * 4);
    const int64_t cap = (int64_t)device_num_sms() * 8;
    const unsigned grid = (unsigned)(blocks < cap || cap <= 0 ? blocks : cap);
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    if (!row_src && ldx == cols)
      amax_rows_kernel<true><<<grid, 256, 0, s>>>(xb, rows, cols, ldx, row_src, amax_bits);
    else
      amax_rows_kernel<false><<<grid, 256, 0, s>>>(xb, rows, cols, ldx, row_src, amax_bits);
  }
  return launch_status();
}

}  // namespace
}  // namespace nvfp4moe

using namespace nvfp4moe;

extern "C" size_t nvfp4_quantize_workspace_size(void) { return 256; }

extern "C" size_t moe_quantize_dispatch_workspace_size(int E) {
  if (E < 1) return 0;
  return 256 + (size_t)ceil_div((int64_t)(E + 1) * 4, 256) * 256;
}

extern "C" int nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                              const float* gs_in, float* gs_out, const int32_t* row_src,
                              uint8_t* codes, uint8_t* sf, int sf_layout, void* ws,
                              size_t ws_bytes, void* stream) {
  NVFP4_CHECK(rows >= 0 && cols >= 0 && cols % 16 == 0, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(sf_layout == NVFP4_SF_ROWMAJOR || sf_layout == NVFP4_SF_TILED || sf_layout == NVFP4_SF_TILED_ROWS,
              NVFP4MOE_ERR_INVALID);
  if (rows == 0 || cols == 0) return NVFP4MOE_OK;
  NVFP4_CHECK(x && codes && sf, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(ldx >= cols && ldx % 8 == 0 && aligned(x, 16) && aligned(codes, 8), NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(sf_layout == NVFP4_SF_ROWMAJOR || aligned(sf, 4), NVFP4MOE_ERR_INVALID);
  cudaStream_t s = as_stream(stream);
  uint32_t* amax_bits = nullptr;
  if (!gs_in) {
    NVFP4_CHECK(ws && ws_bytes >= nvfp4_quantize_workspace_size() && aligned(ws, 16),
                NVFP4MOE_ERR_WORKSPACE);
    amax_bits = static_cast<uint32_t*>(ws);
    NVFP4_TRY(launch_amax(x, rows, cols, ldx, row_src, amax_bits, s));
  }
  const int64_t warps = rows * ceil_div(cols, kChunk);
  const int64_t blocks = ceil_div(warps, kWarpsPerBlock);
  NVFP4_CHECK(blocks < (1ll << 31), NVFP4MOE_ERR_UNSUPPORTED);
  quantize_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(x), rows, cols, ldx, gs_in, amax_bits, gs_out, row_src,
      codes, sf, sf_layout);
  return launch_status();
}

namespace nvfp4moe {
int launch_dispatch_quantize(const void* x, int64_t T, int64_t K, int64_t ldx, int k, const float* gs_in,
                             const uint32_t* amax_bits, float* gs_out, const int32_t* topk_ids,
                             const int32_t* offsets, const int32_t* flat_to_perm, const int32_t* pad_off,
                             uint8_t* a_codes, uint8_t* a_sf, cudaStream_t s) {
  if (T == 0) return NVFP4MOE_OK;
  const int64_t warps = T * ceil_div(K, kChunk);
  dispatch_quantize_kernel<<<(unsigned)ceil_div(warps, kWarpsPerBlock), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(x), T, K, ldx, k, gs_in, amax_bits, gs_out, topk_ids, offsets,
      flat_to_perm, pad_off, a_codes, a_sf);
  return launch_status();
}
}  // namespace nvfp4moe

extern "C" int moe_quantize_dispatch(const void* x, int64_t T, int64_t K, int64_t ldx, int k, int E,
                                     const int32_t* topk_ids, const int32_t* offsets,
                                     const int32_t* flat_to_perm, const float* gs_in,
                                     float* gs_out, uint8_t* a_codes, uint8_t* a_sf,
                                     int64_t a_rows, void* ws, size_t ws_bytes, void* stream) {
  NVFP4_CHECK(T >= 0 && K > 0 && K % 64 == 0 && k >= 1 && k <= 16 && E >= 1 && E <= 1024,
              NVFP4MOE_ERR_UNSUPPORTED);
  NVFP4_CHECK(x && topk_ids && offsets && flat_to_perm && a_codes && a_sf, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(ldx >= K && ldx % 8 == 0 && aligned(x, 16) && aligned(a_codes, 8) && aligned(a_sf, 4),
              NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(a_rows >= nvfp4moe_padded_rows(T * k, E), NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(ws && ws_bytes >= moe_quantize_dispatch_workspace_size(E) && aligned(ws, 16),
              NVFP4MOE_ERR_WORKSPACE);
  cudaStream_t s = as_stream(stream);
  uint32_t* amax_bits = static_cast<uint32_t*>(ws);
  int32_t* pad_off = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + 256);
  padded_offsets_kernel<<<1, 32, 0, s>>>(offsets, E, pad_off);
  NVFP4_TRY(launch_status());
  if (T == 0) return NVFP4MOE_OK;
  if (!gs_in) NVFP4_TRY(launch_amax(x, T, K, ldx, nullptr, amax_bits, s));
  return launch_dispatch_quantize(x, T, K, ldx, k, gs_in, gs_in ? nullptr : amax_bits, gs_out, topk_ids, offsets,
                                  flat_to_perm, pad_off, a_codes, a_sf, s);
}

extern "C" int nvfp4_rmsnorm_rope_quantize(const void* x, int64_t rows, int64_t D, int64_t ldx,
                                           const float* gamma, float eps, int64_t rope_dims,
                                           const int32_t* positions, const float* cos_tab,
                                           const float* sin_tab, int64_t max_pos, const float* gs,
                                           uint8_t* codes, uint8_t* sf, int sf_layout, float* y_out,
                                           void* stream) {
  NVFP4_CHECK(rows >= 0 && D > 0 && D % 16 == 0 && rope_dims >= 0 && rope_dims % 16 == 0 && rope_dims <= D,
              NVFP4MOE_ERR_UNSUPPORTED);
  NVFP4_CHECK(sf_layout == NVFP4_SF_ROWMAJOR || sf_layout == NVFP4_SF_TILED || sf_layout == NVFP4_SF_TILED_ROWS,
              NVFP4MOE_ERR_INVALID);
  if (rows == 0) return NVFP4MOE_OK;
  NVFP4_CHECK(x && gamma && gs && codes && sf && eps >= 0.0f, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(rope_dims == 0 || (positions && cos_tab && sin_tab && max_pos > 0), NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(ldx >= D && ldx % 8 == 0 && aligned(x, 16) && aligned(codes, 8) && aligned(sf, 4) &&
                  aligned(gamma, 16) && (!y_out || aligned(y_out, 16)) &&
                  (rope_dims == 0 || (aligned(cos_tab, 16) && aligned(sin_tab, 16))),
              NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(rows * 32 < (1ll << 40), NVFP4MOE_ERR_UNSUPPORTED);
  int* status = device_status_word();
  NVFP4_CHECK(status, NVFP4MOE_ERR_LAUNCH);
  NormRopeArgs a{static_cast<const __nv_bfloat16*>(x), rows, D, ldx, gamma, eps, rope_dims, positions,
                 cos_tab, sin_tab, max_pos, gs, codes, sf, sf_layout, y_out, status};
  cudaStream_t s = as_stream(stream);
  // lane groups of G lanes with up to BPL blocks each: G * BPL covers the row
  const int64_t nb = D / 16;
  if (nb <= 4) launch_norm_rope<4, 1>(a, s);
  else if (nb <= 8) launch_norm_rope<4, 2>(a, s);
  else if (nb <= 12) launch_norm_rope<4, 3>(a, s);
  else if (nb <= 24) launch_norm_rope<8, 3>(a, s);
  else if (nb <= 48) launch_norm_rope<16, 3>(a, s);
  else if (nb <= 96) launch_norm_rope<32, 3>(a, s);
  else norm_rope_quantize_long_kernel<<<(unsigned)ceil_div(rows, 8), 256, 0, s>>>(a);
  return launch_status();
}
