// Routing, permutation and combine kernels of the MoE forward
// ("NVFP4 MegaMoE Kernel" README, "MoE Runner" steps 1 and 6, and
// "Correctness Bugs Fixed" bug 5: expert counts by bincount).
//
// Permutation (stable counting sort of the T*k flat slots by expert):
//   1. count:   per chunk of kPermChunk slots, a shared-memory histogram
//               -> counts[chunk][e]
//   2. scan:    one block: per expert, exclusive sum over chunks, then an
//               exclusive sum over experts -> offsets and the first row of
//               every (chunk, expert) pair
//   3. scatter: per chunk, one warp walks the slots in order 32 at a time;
//               __match_any_sync groups equal experts inside the warp, and
//               the rank among lower lanes gives the stable position.
// Up to kPermChunk slots, one block does all three (perm_single_kernel).
#include "common.cuh"

#include <mutex>

namespace nvfp4moe {
namespace {

constexpr int kPermChunk = 1024;

// One warp per token; each lane holds VPL logits (expert lane + 32*i).
template <int VPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits,
                                                         int64_t T, int E, int k,
                                                         int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int64_t t = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  int my_i;
  float my_w;
  route_token<VPL>(logits + t * E, E, k, lane, my_i, my_w);
  if (lane < k) {
    ids[t * k + lane] = my_i;
    w[t * k + lane] = my_w;
  }
}

__global__ void __launch_bounds__(256) perm_count_kernel(const int32_t* __restrict__ ids, int64_t n,
                                                         int E, int32_t* __restrict__ counts) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t f0 = blockIdx.x * (int64_t)kPermChunk;
  for (int i = threadIdx.x; i < kPermChunk; i += blockDim.x) {
    const int64_t f = f0 + i;
    if (f < n) atomicAdd(&hist[ids[f]], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[blockIdx.x * (int64_t)E + e] = hist[e];
}

// One block of 1024 threads; thread e owns expert e (E <= 1024).
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ counts, int nchunk,
                                                         int E, int64_t n,
                                                         int32_t* __restrict__ offsets) {
  __shared__ int32_t warp_sums[32];
  const int e = threadIdx.x;
  int total = 0;
  // the chunks' counts of expert e become exclusive prefixes; 16 loads are in
  // flight at a time (one at a time, the loop was a chain of L2 round trips)
  if (e < E) {
    for (int c0 = 0; c0 < nchunk; c0 += 16) {
      int v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = c0 + j < nchunk ? counts[(int64_t)(c0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (c0 + j < nchunk) counts[(int64_t)(c0 + j) * E + e] = total;
        total += v[j];
      }
    }
  }
  // block-wide exclusive scan of the per-expert totals
  const int lane = e & 31, wid = e >> 5;
  int incl = total;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, si, d);
      if (lane >= d) si += y;
    }
    warp_sums[lane] = si - s;
  }
  __syncthreads();
  const int excl = warp_sums[wid] + incl - total;
  if (e < E) {
    offsets[e] = excl;
    for (int c0 = 0; c0 < nchunk; c0 += 16) {
      int v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = c0 + j < nchunk ? counts[(int64_t)(c0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + j < nchunk) counts[(int64_t)(c0 + j) * E + e] = v[j] + excl;
    }
  }
  if (e == 0) offsets[E] = (int32_t)n;
}

__global__ void __launch_bounds__(32) perm_scatter_kernel(const int32_t* __restrict__ ids, int64_t n,
                                                          int E, const int32_t* __restrict__ base,
                                                          int32_t* __restrict__ perm_to_flat,
                                                          int32_t* __restrict__ flat_to_perm) {
  extern __shared__ int32_t next[];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) next[e] = base[blockIdx.x * (int64_t)E + e];
  const int64_t f0 = blockIdx.x * (int64_t)kPermChunk;
  // the chunk's experts are all loaded up front: the ordered walk below is
  // then a chain of shared-memory and warp operations, not of global loads
  int ev[kPermChunk / 32];
#pragma unroll
  for (int i = 0; i < kPermChunk / 32; ++i) {
    const int64_t f = f0 + 32 * i + lane;
    ev[i] = f < n ? ids[f] : -1 - lane;  // invalid lanes never match a real expert
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < kPermChunk / 32; ++i) {
    const int64_t f = f0 + 32 * i + lane;
    const bool valid = f < n;
    const int e = ev[i];
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int start = valid ? next[e] : 0;
    __syncwarp();
    if (valid) {
      const int pos = start + rank;
      perm_to_flat[pos] = (int32_t)f;
      flat_to_perm[f] = pos;
      if (lane == 31 - __clz(peers)) next[e] = start + __popc(peers);
    }
    __syncwarp();
  }
}

// n <= kPermChunk slots (decode-sized batches): the three steps in one block
// of 1024 threads, the launch that dominates them at this size paid once: a
// shared-memory histogram, the exclusive sum over experts (thread e owns
// expert e), then warp 0 walks the slots in order as perm_scatter_kernel does.
__global__ void __launch_bounds__(1024) perm_single_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ perm_to_flat,
                                                           int32_t* __restrict__ flat_to_perm) {
  __shared__ int32_t next[1024];
  __shared__ int32_t slot_e[kPermChunk];
  __shared__ int32_t warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid < E) next[tid] = 0;
  __syncthreads();
  if (tid < n) {
    const int e = ids[tid];
    slot_e[tid] = e;
    atomicAdd(&next[e], 1);
  }
  __syncthreads();
  const int total = tid < E ? next[tid] : 0;
  int incl = total;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, si, d);
      if (lane >= d) si += y;
    }
    warp_sums[lane] = si - s;
  }
  __syncthreads();
  const int excl = warp_sums[wid] + incl - total;
  if (tid < E) {
    offsets[tid] = excl;
    next[tid] = excl;
  }
  if (tid == 0) offsets[E] = n;
  __syncthreads();
  if (wid == 0) {
    for (int i = 0; i < n; i += 32) {
      const int f = i + lane;
      const bool valid = f < n;
      const int e = valid ? slot_e[f] : -1 - lane;  // invalid lanes never match a real expert
      const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int start = valid ? next[e] : 0;
      __syncwarp();
      if (valid) {
        const int pos = start + rank;
        perm_to_flat[pos] = f;
        flat_to_perm[f] = pos;
        if (lane == 31 - __clz(peers)) next[e] = start + __popc(peers);
      }
      __syncwarp();
    }
  }
}

constexpr int kCombineCols = 1024;   // columns per block: 128 threads x 8

__global__ void __launch_bounds__(128) combine_kernel(const __nv_bfloat16* __restrict__ out,
                                                      int64_t ldo, const float* __restrict__ w,
                                                      const int32_t* __restrict__ flat_to_perm,
                                                      int k, int64_t K,
                                                      __nv_bfloat16* __restrict__ y, int64_t ldy) {
  __shared__ int64_t row[16];
  __shared__ float wt[16];
  // block (t, part): token t, columns [part * kCombineCols, (part + 1) * kCombineCols)
  const int64_t t = blockIdx.x;
  if (threadIdx.x < k) {
    row[threadIdx.x] = flat_to_perm[t * k + threadIdx.x];
    wt[threadIdx.x] = w[t * k + threadIdx.x];
  }
  __syncthreads();
  const int64_t c_end = min(K, (int64_t)(blockIdx.y + 1) * kCombineCols);
  for (int64_t c = (int64_t)blockIdx.y * kCombineCols + threadIdx.x * 8; c < c_end; c += blockDim.x * 8) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(out + row[j] * ldo + c));
      float f[8];
      bf16x8_to_f32(u, f);
      const float wj = wt[j];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, f[i], acc[i]);
    }
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      p[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(y + t * ldy + c) = make_uint4(p[0], p[1], p[2], p[3]);
  }
}

}  // namespace
}  // namespace nvfp4moe

using namespace nvfp4moe;

extern "C" int moe_route_topk(const float* logits, int64_t T, int E, int k, int32_t* topk_ids,
                              float* topk_w, void* stream) {
  NVFP4_CHECK(T >= 0 && k >= 1 && k <= 16 && E >= k && E <= 1024, NVFP4MOE_ERR_UNSUPPORTED);
  if (T == 0) return NVFP4MOE_OK;
  NVFP4_CHECK(logits && topk_ids && topk_w, NVFP4MOE_ERR_INVALID);
  cudaStream_t s = as_stream(stream);
  const unsigned blocks = (unsigned)ceil_div(T, 8);
  const int vpl = (E + 31) / 32;
  if (vpl <= 1) route_topk_kernel<1><<<blocks, 256, 0, s>>>(logits, T, E, k, topk_ids, topk_w);
  else if (vpl <= 2) route_topk_kernel<2><<<blocks, 256, 0, s>>>(logits, T, E, k, topk_ids, topk_w);
  else if (vpl <= 4) route_topk_kernel<4><<<blocks, 256, 0, s>>>(logits, T, E, k, topk_ids, topk_w);
  else if (vpl <= 8) route_topk_kernel<8><<<blocks, 256, 0, s>>>(logits, T, E, k, topk_ids, topk_w);
  else if (vpl <= 16) route_topk_kernel<16><<<blocks, 256, 0, s>>>(logits, T, E, k, topk_ids, topk_w);
  else route_topk_kernel<32><<<blocks, 256, 0, s>>>(logits, T, E, k, topk_ids, topk_w);
  return launch_status();
}

extern "C" size_t moe_permute_workspace_size(int64_t T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return 0;
  const int64_t nchunk = ceil_div(T * k, kPermChunk);
  return (size_t)ceil_div((nchunk > 0 ? nchunk : 1) * E * 4, 256) * 256;
}

extern "C" int moe_permute(const int32_t* topk_ids, int64_t T, int k, int E, int32_t* offsets,
                           int32_t* perm_to_flat, int32_t* flat_to_perm, void* ws, size_t ws_bytes,
                           void* stream) {
  NVFP4_CHECK(T >= 0 && k >= 1 && k <= 16 && E >= 1 && E <= 1024, NVFP4MOE_ERR_UNSUPPORTED);
  NVFP4_CHECK(T * k < (1ll << 31), NVFP4MOE_ERR_UNSUPPORTED);
  NVFP4_CHECK(offsets, NVFP4MOE_ERR_INVALID);
  const int64_t n = T * k;
  NVFP4_CHECK(n == 0 || (topk_ids && perm_to_flat && flat_to_perm), NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(ws && ws_bytes >= moe_permute_workspace_size(T, k, E) && aligned(ws, 16),
              NVFP4MOE_ERR_WORKSPACE);
  cudaStream_t s = as_stream(stream);
  if (n <= kPermChunk) {
    perm_single_kernel<<<1, 1024, 0, s>>>(topk_ids, (int)n, E, offsets, perm_to_flat, flat_to_perm);
    return launch_status();
  }
  const int nchunk = (int)ceil_div(n, kPermChunk);
  int32_t* counts = static_cast<int32_t*>(ws);
  if (nchunk > 0)
    perm_count_kernel<<<nchunk, 256, E * sizeof(int32_t), s>>>(topk_ids, n, E, counts);
  perm_scan_kernel<<<1, 1024, 0, s>>>(counts, nchunk, E, n, offsets);
  if (nchunk > 0)
    perm_scatter_kernel<<<nchunk, 32, E * sizeof(int32_t), s>>>(topk_ids, n, E, counts,
                                                                 perm_to_flat, flat_to_perm);
  return launch_status();
}

extern "C" int moe_combine(const void* out, int64_t ldo, const float* topk_w,
                           const int32_t* flat_to_perm, int64_t T, int k, int64_t K, void* y,
                           int64_t ldy, void* stream) {
  NVFP4_CHECK(T >= 0 && k >= 1 && k <= 16 && K >= 0 && K % 8 == 0, NVFP4MOE_ERR_UNSUPPORTED);
  if (T == 0 || K == 0) return NVFP4MOE_OK;
  NVFP4_CHECK(out && topk_w && flat_to_perm && y, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(ldo >= K && ldy >= K && ldo % 8 == 0 && ldy % 8 == 0 && aligned(out, 16) &&
                  aligned(y, 16),
              NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(T < (1ll << 31) && ceil_div(K, kCombineCols) <= 65535, NVFP4MOE_ERR_UNSUPPORTED);
  combine_kernel<<<dim3((unsigned)T, (unsigned)ceil_div(K, kCombineCols)), 128, 0, as_stream(stream)>>>(
      static_cast<const __nv_bfloat16*>(out), ldo, topk_w, flat_to_perm, k, K,
      static_cast<__nv_bfloat16*>(y), ldy);
  return launch_status();
}

// ------------------------------------------------------------------ permutation without workspace
//
// moe_permute_static_ws: the same three kernels as moe_permute, with their
// per-chunk count table in a fixed device array that the library owns,
// instead of in caller-provided workspace. It exists for callers that cannot
// allocate device memory at the point of the call -- for example code that
// runs inside another framework's execution callback whose contract forbids
// allocation, or latency-critical paths that must not risk the implicit
// device synchronisation an allocation can cause -- and that have no spare
// workspace to hand in.

namespace {

// ceil(T*k / 1024) * E count entries: 1 MiB of int32. Every GPU that loads
// this library keeps this array until the process exits.
constexpr int64_t kStaticPermScratchInts = 262144;
static __device__ __align__(256) int32_t g_static_perm_scratch[kStaticPermScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_static_perm_mutex;
int32_t* g_static_perm_addr[kMaxDevices] = {};

// Device address of the array on the current device. In host code the array's
// name only stands in for it, so the address is looked up (once per device,
// with that device current) and handed to the kernels as an ordinary pointer.
int32_t* static_perm_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_static_perm_mutex);
  if (!g_static_perm_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_perm_scratch) != cudaSuccess) return nullptr;
    g_static_perm_addr[dev] = static_cast<int32_t*>(p);
  }
  return g_static_perm_addr[dev];
}

}  // namespace

extern "C" int moe_permute_static_ws(const int32_t* topk_ids, int64_t T, int k, int E,
                                     int32_t* offsets, int32_t* perm_to_flat,
                                     int32_t* flat_to_perm, void* stream) {
  NVFP4_CHECK(T >= 0 && k >= 1 && k <= 16 && E >= 1 && E <= 1024, NVFP4MOE_ERR_UNSUPPORTED);
  NVFP4_CHECK(T * k < (1ll << 31), NVFP4MOE_ERR_UNSUPPORTED);
  const int64_t n = T * k;
  const int64_t nchunk = ceil_div(n, kPermChunk);
  // the count table needs nchunk * E entries of the fixed array
  NVFP4_CHECK(nchunk * E <= kStaticPermScratchInts, NVFP4MOE_ERR_WORKSPACE);
  NVFP4_CHECK(offsets, NVFP4MOE_ERR_INVALID);
  NVFP4_CHECK(n == 0 || (topk_ids && perm_to_flat && flat_to_perm), NVFP4MOE_ERR_INVALID);
  cudaStream_t s = as_stream(stream);
  if (n <= kPermChunk) {
    perm_single_kernel<<<1, 1024, 0, s>>>(topk_ids, (int)n, E, offsets, perm_to_flat, flat_to_perm);
    return launch_status();
  }
  int32_t* counts = static_perm_scratch();
  NVFP4_CHECK(counts != nullptr, NVFP4MOE_ERR_LAUNCH);
  // every entry the scan reads is written by the count kernel first, so the
  // array needs no clearing between calls
  if (nchunk > 0)
    perm_count_kernel<<<(unsigned)nchunk, 256, E * sizeof(int32_t), s>>>(topk_ids, n, E, counts);
  perm_scan_kernel<<<1, 1024, 0, s>>>(counts, (int)nchunk, E, n, offsets);
  if (nchunk > 0)
    perm_scatter_kernel<<<(unsigned)nchunk, 32, E * sizeof(int32_t), s>>>(topk_ids, n, E, counts,
                                                                         perm_to_flat, flat_to_perm);
  return launch_status();
}
