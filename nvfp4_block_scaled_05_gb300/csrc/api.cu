// Host-side entry points: sizes and layouts, and moe_forward, which enqueues
// the six stages of the "NVFP4 MegaMoE Kernel" README "MoE Runner" (with the
// fused L1 of "Fused SwiGLU - How It Works") on one stream.
#include "common.cuh"

using namespace nvfp4moe;

extern "C" const char* nvfp4moe_status_string(int status) {
  switch (status) {
    case NVFP4MOE_OK: return "ok";
    case NVFP4MOE_ERR_INVALID: return "invalid argument";
    case NVFP4MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case NVFP4MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4MOE_ERR_LAUNCH: return "CUDA launch error";
    case NVFP4MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

extern "C" size_t nvfp4_sf_bytes(int64_t rows, int64_t cols, int sf_layout) {
  if (rows < 0 || cols < 0) return 0;
  if (sf_layout == NVFP4_SF_ROWMAJOR) return (size_t)(rows * (cols / 16));
  if (sf_layout == NVFP4_SF_TILED) return (size_t)(ceil_div(rows, 128) * ceil_div(cols, 64) * 512);
  if (sf_layout == NVFP4_SF_TILED_ROWS) return (size_t)(ceil_div(rows, 128) * ceil_div(cols, 256) * 2048);
  return 0;
}

extern "C" int64_t nvfp4moe_padded_rows(int64_t M, int E) {
  if (M < 0 || E < 1) return 0;
  const int64_t groups = M < E ? M : E;
  const int64_t r = ceil_div(M + groups * 127, 128) * 128;
  return r > 128 ? r : 128;
}

extern "C" int nvfp4moe_interleave_row_map(int64_t two_i, int32_t* map_host) {
  if (two_i <= 0 || two_i % 16 != 0 || !map_host) return NVFP4MOE_ERR_INVALID;
  const int64_t I = two_i / 2;
  for (int64_t n = 0; n < I; ++n) {
    const int64_t base = 16 * (n / 8) + n % 8;
    map_host[base] = (int32_t)n;          // gate row n
    map_host[base + 8] = (int32_t)(I + n);  // up row n
  }
  return NVFP4MOE_OK;
}

namespace {

struct Layout {
  int64_t off[12];
  int64_t total;
};

int64_t up256(int64_t v) { return ceil_div(v, 256) * 256; }

// topk_ids, topk_w, offsets, perm_to_flat, flat_to_perm, gs_x, a_codes, a_sf,
// h_codes, h_sf, out, then the permute and dispatch scratch.
Layout make_layout(int64_t T, int64_t K, int64_t I, int E, int k) {
  Layout L{};
  const int64_t M = T * k;
  const int64_t a_rows = nvfp4moe_padded_rows(M, E);
  int64_t o = 0;
  auto take = [&](int64_t bytes) {
    const int64_t at = o;
    o += up256(bytes > 0 ? bytes : 1);
    return at;
  };
  L.off[0] = take(M * 4);
  L.off[1] = take(M * 4);
  L.off[2] = take((E + 1) * 4);
  L.off[3] = take(M * 4);
  L.off[4] = take(M * 4);
  L.off[5] = take(4);
  L.off[6] = take(a_rows * (K / 2));
  L.off[7] = take((int64_t)nvfp4_sf_bytes(a_rows, K, NVFP4_SF_TILED_ROWS));
  L.off[8] = take(a_rows * (I / 2));
  L.off[9] = take((int64_t)nvfp4_sf_bytes(a_rows, I, NVFP4_SF_TILED_ROWS));
  L.off[10] = take(M * K * 2);
  L.off[11] = a_rows;
  // scratch: the permute and dispatch workspaces (moe_forward), or the fused
  // front's (moe_forward_static), whichever is larger
  const int64_t split = up256((int64_t)moe_permute_workspace_size(T, k, E)) +
                        up256((int64_t)moe_quantize_dispatch_workspace_size(E));
  const int64_t front = (int64_t)front_workspace_bytes(T, E);
  take(split > front ? split : front);
  L.total = o;
  return L;
}

bool forward_shape_ok(int64_t T, int64_t K, int64_t I, int E, int k) {
  return T >= 0 && K > 0 && K % 128 == 0 && I > 0 && I % 64 == 0 && k >= 1 && k <= 16 && E >= k &&
         E <= 1024 && T * k < (1ll << 31);
}

}  // namespace

extern "C" size_t moe_forward_workspace_size(int64_t T, int64_t K, int64_t I, int E, int k) {
  if (!forward_shape_ok(T, K, I, E, k)) return 0;
  return (size_t)make_layout(T, K, I, E, k).total;
}

extern "C" int moe_forward_workspace_layout(int64_t T, int64_t K, int64_t I, int E, int k,
                                            int64_t* offs_host) {
  if (!forward_shape_ok(T, K, I, E, k)) return NVFP4MOE_ERR_UNSUPPORTED;
  if (!offs_host) return NVFP4MOE_ERR_INVALID;
  const Layout L = make_layout(T, K, I, E, k);
  for (int i = 0; i < 12; ++i) offs_host[i] = L.off[i];
  return NVFP4MOE_OK;
}

extern "C" int moe_forward(const void* x, const float* router_logits, int64_t T, int64_t K,
                           int64_t I, int E, int k, const uint8_t* w1_codes, const uint8_t* w1_sf,
                           const float* gs_w1, const uint8_t* w2_codes, const uint8_t* w2_sf,
                           const float* gs_w2, const float* gs_h, void* y, void* ws,
                           size_t ws_bytes, void* stream) {
  NVFP4_CHECK(forward_shape_ok(T, K, I, E, k), NVFP4MOE_ERR_UNSUPPORTED);
  if (T == 0) return NVFP4MOE_OK;
  NVFP4_CHECK(x && router_logits && w1_codes && w1_sf && gs_w1 && w2_codes && w2_sf && gs_w2 &&
                  gs_h && y,
              NVFP4MOE_ERR_INVALID);
  const Layout L = make_layout(T, K, I, E, k);
  NVFP4_CHECK(ws && ws_bytes >= (size_t)L.total && aligned(ws, 256), NVFP4MOE_ERR_WORKSPACE);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* ids = reinterpret_cast<int32_t*>(w + L.off[0]);
  float* topw = reinterpret_cast<float*>(w + L.off[1]);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.off[2]);
  int32_t* p2f = reinterpret_cast<int32_t*>(w + L.off[3]);
  int32_t* f2p = reinterpret_cast<int32_t*>(w + L.off[4]);
  float* gs_x = reinterpret_cast<float*>(w + L.off[5]);
  uint8_t* a_codes = w + L.off[6];
  uint8_t* a_sf = w + L.off[7];
  uint8_t* h_codes = w + L.off[8];
  uint8_t* h_sf = w + L.off[9];
  void* out = w + L.off[10];
  const int64_t a_rows = L.off[11];
  const int64_t M = T * k;
  uint8_t* scratch = w + L.off[10] + up256(M * K * 2);
  if (moe_forward_uses_fused_dispatch(T, E, k)) {
    // stages 1-2 in one cooperative kernel, the global scale of x computed in it
    const size_t front_bytes = (size_t)(L.total - (L.off[10] + up256(M * K * 2)));
    NVFP4_TRY(moe_dispatch(x, K, router_logits, T, K, E, k, gs_x, ids, topw, offsets, p2f, f2p, a_codes,
                           a_sf, a_rows, scratch, front_bytes, stream));
  } else {
    uint8_t* perm_ws = scratch;
    const size_t perm_bytes = moe_permute_workspace_size(T, k, E);
    uint8_t* disp_ws = perm_ws + up256((int64_t)perm_bytes);
    const size_t disp_bytes = moe_quantize_dispatch_workspace_size(E);
    NVFP4_TRY(moe_route_topk(router_logits, T, E, k, ids, topw, stream));
    NVFP4_TRY(moe_permute(ids, T, k, E, offsets, p2f, f2p, perm_ws, perm_bytes, stream));
    NVFP4_TRY(moe_quantize_dispatch(x, T, K, K, k, E, ids, offsets, f2p, nullptr, gs_x, a_codes, a_sf,
                                    a_rows, disp_ws, disp_bytes, stream));
  }
  NVFP4_TRY(nvfp4_grouped_gemm_swiglu(a_codes, a_sf, gs_x, a_rows, w1_codes, w1_sf, gs_w1, offsets,
                                      E, I, K, gs_h, h_codes, h_sf, stream));
  NVFP4_TRY(nvfp4_grouped_gemm(h_codes, h_sf, gs_h, a_rows, w2_codes, w2_sf, gs_w2, offsets, E, K,
                               I, out, K, stream));
  NVFP4_TRY(moe_combine(out, K, topw, f2p, T, k, K, y, K, stream));
  return NVFP4MOE_OK;
}

extern "C" int moe_forward_static(const void* x, const float* router_logits, int64_t T, int64_t K,
                                  int64_t I, int E, int k, const float* gs_x, const uint8_t* w1_codes,
                                  const uint8_t* w1_sf, const float* gs_w1, const uint8_t* w2_codes,
                                  const uint8_t* w2_sf, const float* gs_w2, const float* gs_h, void* y,
                                  void* ws, size_t ws_bytes, void* stream) {
  NVFP4_CHECK(forward_shape_ok(T, K, I, E, k), NVFP4MOE_ERR_UNSUPPORTED);
  if (T == 0) return NVFP4MOE_OK;
  NVFP4_CHECK(x && router_logits && gs_x && w1_codes && w1_sf && gs_w1 && w2_codes && w2_sf && gs_w2 &&
                  gs_h && y && aligned(x, 16),
              NVFP4MOE_ERR_INVALID);
  const Layout L = make_layout(T, K, I, E, k);
  NVFP4_CHECK(ws && ws_bytes >= (size_t)L.total && aligned(ws, 256), NVFP4MOE_ERR_WORKSPACE);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* ids = reinterpret_cast<int32_t*>(w + L.off[0]);
  float* topw = reinterpret_cast<float*>(w + L.off[1]);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.off[2]);
  int32_t* p2f = reinterpret_cast<int32_t*>(w + L.off[3]);
  int32_t* f2p = reinterpret_cast<int32_t*>(w + L.off[4]);
  uint8_t* a_codes = w + L.off[6];
  uint8_t* a_sf = w + L.off[7];
  uint8_t* h_codes = w + L.off[8];
  uint8_t* h_sf = w + L.off[9];
  void* out = w + L.off[10];
  const int64_t a_rows = L.off[11];
  const int64_t M = T * k;
  uint8_t* front_ws = w + L.off[10] + up256(M * K * 2);
  const size_t front_bytes = (size_t)(L.total - (L.off[10] + up256(M * K * 2)));
  NVFP4_TRY(moe_dispatch_static(x, K, router_logits, T, K, E, k, gs_x, ids, topw, offsets, p2f, f2p,
                                a_codes, a_sf, a_rows, front_ws, front_bytes, stream));
  NVFP4_TRY(nvfp4_grouped_gemm_swiglu(a_codes, a_sf, gs_x, a_rows, w1_codes, w1_sf, gs_w1, offsets,
                                      E, I, K, gs_h, h_codes, h_sf, stream));
  NVFP4_TRY(nvfp4_grouped_gemm(h_codes, h_sf, gs_h, a_rows, w2_codes, w2_sf, gs_w2, offsets, E, K,
                               I, out, K, stream));
  NVFP4_TRY(moe_combine(out, K, topw, f2p, T, k, K, y, K, stream));
  return NVFP4MOE_OK;
}

extern "C" size_t moe_dispatch_static_workspace_size(int64_t T, int E) {
  if (T < 1 || E < 1 || E > 1024) return 0;
  return front_workspace_bytes(T, E);
}

extern "C" int moe_dispatch_static(const void* x, int64_t ldx, const float* router_logits, int64_t T,
                                   int64_t K, int E, int k, const float* gs_x, int32_t* topk_ids,
                                   float* topk_w, int32_t* offsets, int32_t* perm_to_flat,
                                   int32_t* flat_to_perm, uint8_t* a_codes, uint8_t* a_sf,
                                   int64_t a_rows, void* ws, size_t ws_bytes, void* stream) {
  NVFP4_CHECK(T >= 0 && K > 0 && K % 64 == 0 && k >= 1 && k <= 16 && E >= k && E <= 1024 &&
                  T * k < (1ll << 31),
              NVFP4MOE_ERR_UNSUPPORTED);
  if (T == 0) return NVFP4MOE_OK;
  NVFP4_CHECK(x && router_logits && gs_x && topk_ids && topk_w && offsets && perm_to_flat &&
                  flat_to_perm && a_codes && a_sf,
              NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(ldx >= K && ldx % 8 == 0 && aligned(x, 16) && aligned(a_codes, 8) && aligned(a_sf, 4),
              NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(a_rows >= nvfp4moe_padded_rows(T * k, E), NVFP4MOE_ERR_INVALID);
  return moe_front(x, ldx, router_logits, T, K, E, k, gs_x, nullptr, topk_ids, topk_w, offsets, perm_to_flat,
                   flat_to_perm, a_codes, a_sf, ws, ws_bytes, as_stream(stream));
}

extern "C" int moe_dispatch_supported(int64_t T, int E, int k) { return moe_front_fits(T, E, k) ? 1 : 0; }

// Measured on GB300: the fused dispatch (with its quantize + scatter as a
// second kernel above NVFP4MOE_FRONT_FUSED_QUANTIZE_MAX_ROWS routed rows) is
// faster than the separate route/permute/quantize at every size measured
// (1024 rows: 20 against 36 us; 32768 rows: 63 against 89 us; 65536 rows:
// 122 against 147 us; 131072 rows: 224 against 250 us).
extern "C" int moe_forward_uses_fused_dispatch(int64_t T, int E, int k) {
  return T >= 1 && moe_front_fits(T, E, k) ? 1 : 0;
}

extern "C" int moe_dispatch(const void* x, int64_t ldx, const float* router_logits, int64_t T, int64_t K,
                            int E, int k, float* gs_out, int32_t* topk_ids, float* topk_w, int32_t* offsets,
                            int32_t* perm_to_flat, int32_t* flat_to_perm, uint8_t* a_codes, uint8_t* a_sf,
                            int64_t a_rows, void* ws, size_t ws_bytes, void* stream) {
  NVFP4_CHECK(T >= 0 && K > 0 && K % 64 == 0 && k >= 1 && k <= 16 && E >= k && E <= 1024 &&
                  T * k < (1ll << 31),
              NVFP4MOE_ERR_UNSUPPORTED);
  if (T == 0) return NVFP4MOE_OK;
  NVFP4_CHECK(x && router_logits && gs_out && topk_ids && topk_w && offsets && perm_to_flat &&
                  flat_to_perm && a_codes && a_sf,
              NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(ldx >= K && ldx % 8 == 0 && aligned(x, 16) && aligned(a_codes, 8) && aligned(a_sf, 4),
              NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(a_rows >= nvfp4moe_padded_rows(T * k, E), NVFP4MOE_ERR_INVALID);
  return moe_front(x, ldx, router_logits, T, K, E, k, nullptr, gs_out, topk_ids, topk_w, offsets, perm_to_flat,
                   flat_to_perm, a_codes, a_sf, ws, ws_bytes, as_stream(stream));
}

// ------------------------------------------------------------------ single linear

namespace {
__global__ void linear_bounds_kernel(int32_t* bounds, int32_t M) {
  bounds[0] = 0;
  bounds[1] = M;
}
}  // namespace

extern "C" size_t nvfp4_linear_workspace_size(void) { return 256; }

extern "C" int nvfp4_linear(const uint8_t* a_codes, const uint8_t* a_sf, const float* gs_a, int64_t M,
                            int64_t a_rows, const uint8_t* w_codes, const uint8_t* w_sf,
                            const float* gs_w, int64_t N, int64_t K, void* c, int64_t ldc, void* ws,
                            size_t ws_bytes, void* stream) {
  NVFP4_CHECK(M >= 0 && M < (1ll << 31), NVFP4MOE_ERR_UNSUPPORTED);
  if (M == 0) return NVFP4MOE_OK;
  NVFP4_CHECK(a_rows >= ceil_div(M, 128) * 128, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(ws && ws_bytes >= nvfp4_linear_workspace_size() && aligned(ws, 16), NVFP4MOE_ERR_WORKSPACE);
  cudaStream_t s = as_stream(stream);
  int32_t* bounds = static_cast<int32_t*>(ws);
  linear_bounds_kernel<<<1, 1, 0, s>>>(bounds, (int32_t)M);
  NVFP4_TRY(launch_status());
  // one group of M rows: its padded rows are the rows themselves
  return nvfp4_grouped_gemm(a_codes, a_sf, gs_a, a_rows, w_codes, w_sf, gs_w, bounds, 1, N, K, c, ldc,
                            stream);
}
