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
// (atomicMax on the bits orders non-negative floats correctly).
__global__ void __launch_bounds__(256) amax_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                        int64_t rows, int64_t cols, int64_t ldx,
                                                        const int32_t* __restrict__ row_src,
                                                        uint32_t* __restrict__ amax_bits) {
  const int64_t vec_per_row = cols / 8;
  const int64_t total = rows * vec_per_row;
  float m = 0.0f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / vec_per_row, v = i - r * vec_per_row;
    const int64_t src = row_src ? row_src[r] : r;
    if (src < 0) continue;
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(x + src * ldx) + v);
    float f[8];
    bf16x8_to_f32(u, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
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
  uint32_t w0 = 0, w1 = 0, s = 0;
  if (valid) s = quantize_lane16(x + t * ldx, col0, gs, w0, w1);
  const uint32_t word = gather_sf_word(s);
  const int64_t c4 = K / 64;
  for (int j = 0; j < k; ++j) {
    const int64_t f = t * k + j;
    const int e = topk_ids[f];
    const int64_t prow = (int64_t)pad_off[e] + flat_to_perm[f] - offsets[e];
    if (valid) *reinterpret_cast<uint2*>(a_codes + prow * (K / 2) + col0 / 2) = make_uint2(w0, w1);
    if (valid && (lane & 3) == 0)
      *reinterpret_cast<uint32_t*>(a_sf + sf_tiled_offset(prow, col0 / 16, c4)) = word;
  }
}

int launch_amax(const void* x, int64_t rows, int64_t cols, int64_t ldx, const int32_t* row_src,
                uint32_t* amax_bits, cudaStream_t s) {
  if (cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), s) != cudaSuccess) return NVFP4MOE_ERR_LAUNCH;
  const int64_t total = rows * (cols / 8);
  if (total > 0) {
    int64_t blocks = (total + 255) / 256;
    int64_t cap = 4096;
    amax_rows_kernel<<<(unsigned)(blocks < cap ? blocks : cap), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(x), rows, cols, ldx, row_src, amax_bits);
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
  NVFP4_CHECK(sf_layout == NVFP4_SF_ROWMAJOR || sf_layout == NVFP4_SF_TILED, NVFP4MOE_ERR_INVALID);
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
  const int64_t warps = T * ceil_div(K, kChunk);
  dispatch_quantize_kernel<<<(unsigned)ceil_div(warps, kWarpsPerBlock), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(x), T, K, ldx, k, gs_in, gs_in ? nullptr : amax_bits,
      gs_out, topk_ids, offsets, flat_to_perm, pad_off, a_codes, a_sf);
  return launch_status();
}
