// Offline layout helpers ("NVFP4 MegaMoE Kernel" README, "Bridge Layer":
// interleave_l1_weights / deinterleave_l1_weights, assemble_scales_2d_side /
// assemble_scales_3d_side): conversions between row-major scale bytes and the
// two tiled scale layouts the grouped GEMMs read, and the granularity-8
// gate/up row interleave of W1 ("Fused SwiGLU - How It Works"). They run once
// when weights are prepared, so they are plain gather kernels: one thread per
// output byte (scales) or per 16-byte piece of a code row.
#include "common.cuh"

namespace nvfp4moe {
namespace {

// (row, block) of byte o of a tiled scale matrix, or false for a padding byte.
// blocks = cols / 16; c4 = ceil(cols / 64) (TILED), s = ceil(cols / 256) (TILED_ROWS).
__device__ __forceinline__ bool tiled_coords(int64_t o, int layout, int64_t rows, int64_t blocks, int64_t& r,
                                             int64_t& b) {
  if (layout == NVFP4_SF_TILED) {
    const int64_t c4 = (blocks + 3) / 4;
    const int64_t atom = o >> 9, w = o & 511;
    r = (atom / c4) * 128 + ((w & 15) >> 2) * 32 + (w >> 4);
    b = (atom % c4) * 4 + (w & 3);
  } else {
    const int64_t s = (blocks + 15) / 16;
    const int64_t tile = o >> 11, w = o & 2047;
    r = (tile / s) * 128 + (w >> 4);
    b = (tile % s) * 16 + (w & 15);
  }
  return r < rows && b < blocks;
}

__device__ __forceinline__ int64_t tiled_offset(int layout, int64_t r, int64_t b, int64_t blocks) {
  return layout == NVFP4_SF_TILED ? sf_tiled_offset(r, b, (blocks + 3) / 4)
                                  : sf_rows_offset(r, b, (blocks + 15) / 16);
}

// Source row (in the same matrix) of output row q: the granularity-8 gate/up
// interleave (q interleaved, source [gate | up]) or its inverse.
__device__ __forceinline__ int64_t gate_up_src(int64_t q, int64_t inter, int inverse) {
  if (!inverse) {
    const int64_t g = q >> 4, w = q & 15;
    return w < 8 ? 8 * g + w : inter + 8 * g + (w - 8);
  }
  const bool up = q >= inter;
  const int64_t n = up ? q - inter : q;
  return 16 * (n >> 3) + (up ? 8 : 0) + (n & 7);
}

// Every byte of `batch` tiled scale matrices from row-major scales (padding 0).
__global__ void sf_to_tiled_kernel(const uint8_t* __restrict__ src, int64_t rows, int64_t blocks, int layout,
                                   int64_t tiled_bytes, int64_t total, uint8_t* __restrict__ dst) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / tiled_bytes, o = i - m * tiled_bytes;
    int64_t r, b;
    dst[i] = tiled_coords(o, layout, rows, blocks, r, b) ? src[(m * rows + r) * blocks + b] : 0;
  }
}

// Row-major scales of `batch` matrices from tiled ones.
__global__ void sf_from_tiled_kernel(const uint8_t* __restrict__ src, int64_t rows, int64_t blocks, int layout,
                                     int64_t tiled_bytes, int64_t total, uint8_t* __restrict__ dst) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t per = rows * blocks;
    const int64_t m = i / per, rb = i - m * per, r = rb / blocks, b = rb - r * blocks;
    dst[i] = src[m * tiled_bytes + tiled_offset(layout, r, b, blocks)];
  }
}

// One block per output code row: the source row's K/2 bytes, 16 at a time
// when both rows are 16-byte aligned, else byte by byte.
__global__ void gate_up_codes_kernel(const uint8_t* __restrict__ src, int64_t two_i, int64_t row_bytes, int inverse,
                                     int vec16, uint8_t* __restrict__ dst) {
  const int64_t m = blockIdx.y, q = blockIdx.x;
  const int64_t sr = gate_up_src(q, two_i / 2, inverse);
  const uint8_t* s = src + (m * two_i + sr) * row_bytes;
  uint8_t* d = dst + (m * two_i + q) * row_bytes;
  if (vec16) {
    for (int64_t j = threadIdx.x; j < row_bytes / 16; j += blockDim.x)
      reinterpret_cast<uint4*>(d)[j] = reinterpret_cast<const uint4*>(s)[j];
  } else {
    for (int64_t j = threadIdx.x; j < row_bytes; j += blockDim.x) d[j] = s[j];
  }
}

// Every byte of the permuted scale matrices, in layout `layout` (padding bytes
// of a tiled layout are written 0).
__global__ void gate_up_sf_kernel(const uint8_t* __restrict__ src, int64_t two_i, int64_t blocks, int layout,
                                  int64_t mat_bytes, int64_t total, int inverse, uint8_t* __restrict__ dst) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / mat_bytes, o = i - m * mat_bytes;
    int64_t r, b;
    bool valid;
    if (layout == NVFP4_SF_ROWMAJOR) {
      r = o / blocks;
      b = o - r * blocks;
      valid = true;
    } else {
      valid = tiled_coords(o, layout, two_i, blocks, r, b);
    }
    uint8_t v = 0;
    if (valid) {
      const int64_t sr = gate_up_src(r, two_i / 2, inverse);
      v = src[m * mat_bytes + (layout == NVFP4_SF_ROWMAJOR ? sr * blocks + b : tiled_offset(layout, sr, b, blocks))];
    }
    dst[i] = v;
  }
}

int grid_for(int64_t total) {
  const int64_t blocks = (total + 255) / 256;
  const int64_t cap = 8 * (int64_t)(device_num_sms() > 0 ? device_num_sms() : 1);
  return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

int check_sf_args(const void* a, const void* b, int64_t batch, int64_t rows, int64_t cols, int layout) {
  NVFP4_CHECK(batch >= 0 && rows >= 0 && cols >= 0 && cols % 16 == 0, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(layout == NVFP4_SF_TILED || layout == NVFP4_SF_TILED_ROWS, NVFP4MOE_ERR_INVALID);
  if (batch == 0 || rows == 0 || cols == 0) return NVFP4MOE_OK;
  NVFP4_CHECK(a && b, NVFP4MOE_ERR_INVALID);
  return NVFP4MOE_OK;
}

}  // namespace
}  // namespace nvfp4moe

using namespace nvfp4moe;

extern "C" int nvfp4_sf_to_tiled(const uint8_t* sf, int64_t batch, int64_t rows, int64_t cols, int sf_layout,
                                 uint8_t* sf_tiled, void* stream) {
  NVFP4_TRY(check_sf_args(sf, sf_tiled, batch, rows, cols, sf_layout));
  const int64_t per = (int64_t)nvfp4_sf_bytes(rows, cols, sf_layout);
  const int64_t total = batch * per;
  if (total == 0 || rows == 0 || cols == 0) return NVFP4MOE_OK;
  sf_to_tiled_kernel<<<grid_for(total), 256, 0, as_stream(stream)>>>(sf, rows, cols / 16, sf_layout, per, total,
                                                                      sf_tiled);
  return launch_status();
}

extern "C" int nvfp4_sf_from_tiled(const uint8_t* sf_tiled, int64_t batch, int64_t rows, int64_t cols,
                                   int sf_layout, uint8_t* sf, void* stream) {
  NVFP4_TRY(check_sf_args(sf_tiled, sf, batch, rows, cols, sf_layout));
  const int64_t per = (int64_t)nvfp4_sf_bytes(rows, cols, sf_layout);
  const int64_t total = batch * rows * (cols / 16);
  if (total == 0) return NVFP4MOE_OK;
  sf_from_tiled_kernel<<<grid_for(total), 256, 0, as_stream(stream)>>>(sf_tiled, rows, cols / 16, sf_layout, per,
                                                                        total, sf);
  return launch_status();
}

extern "C" int nvfp4_interleave_gate_up(const uint8_t* codes, const uint8_t* sf, int64_t batch, int64_t two_i,
                                        int64_t K, int sf_layout, int inverse, uint8_t* codes_out,
                                        uint8_t* sf_out, void* stream) {
  NVFP4_CHECK(batch >= 0 && two_i >= 0 && two_i % 16 == 0 && K >= 0 && K % 16 == 0, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(sf_layout == NVFP4_SF_ROWMAJOR || sf_layout == NVFP4_SF_TILED || sf_layout == NVFP4_SF_TILED_ROWS,
              NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(inverse == 0 || inverse == 1, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(batch <= 65535 && two_i < (1ll << 31), NVFP4MOE_ERR_UNSUPPORTED);
  if (batch == 0 || two_i == 0 || K == 0) return NVFP4MOE_OK;
  NVFP4_CHECK((codes == nullptr) == (codes_out == nullptr) && (sf == nullptr) == (sf_out == nullptr) &&
                  (codes || sf),
              NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(codes != codes_out || !codes, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(sf != sf_out || !sf, NVFP4MOE_ERR_INVALID);
  cudaStream_t s = as_stream(stream);
  if (codes) {
    const int64_t row_bytes = K / 2;
    const int vec16 = row_bytes % 16 == 0 && aligned(codes, 16) && aligned(codes_out, 16);
    gate_up_codes_kernel<<<dim3((unsigned)two_i, (unsigned)batch), 128, 0, s>>>(codes, two_i, row_bytes, inverse,
                                                                                vec16, codes_out);
    NVFP4_TRY(launch_status());
  }
  if (sf) {
    const int64_t per = (int64_t)nvfp4_sf_bytes(two_i, K, sf_layout);
    const int64_t total = batch * per;
    gate_up_sf_kernel<<<grid_for(total), 256, 0, s>>>(sf, two_i, K / 16, sf_layout, per, total, inverse, sf_out);
    NVFP4_TRY(launch_status());
  }
  return NVFP4MOE_OK;
}
