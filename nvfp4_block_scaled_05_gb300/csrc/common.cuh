// Shared helpers of the sm_103a kernels: NVFP4 block encoding, PTX wrappers
// for mbarrier / TMA / tcgen05, and host-side argument checks.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nvfp4moe.h"

namespace nvfp4moe {

// ------------------------------------------------------------------ host checks

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? NVFP4MOE_OK : NVFP4MOE_ERR_LAUNCH;
}

#define NVFP4_CHECK(cond, code) \
  do {                          \
    if (!(cond)) return (code); \
  } while (0)

#define NVFP4_TRY(expr)             \
  do {                              \
    int _st = (expr);               \
    if (_st != NVFP4MOE_OK) return _st; \
  } while (0)

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Library-wide device state (defined with the GEMM): the device status word
// (int[2]: status, wait site), the bound on every device-side wait, the SM
// count, the failure-path test hook.
int* device_status_word();
uint64_t wait_limit_ns();
int device_num_sms();
int test_stall_on();   // failure-path test hook (nvfp4moe_set_test_stall)

// Fused front (front.cu): routing, permutation, quantization and scatter in
// one cooperative kernel; gs_x null = the global scale is computed from max|x|
// (and written to gs_out when that is not null). moe_front_fits: whether T
// tokens fit its co-resident blocks.
size_t front_workspace_bytes(int64_t T, int E);
bool moe_front_fits(int64_t T, int E, int k);
int moe_front(const void* x, int64_t ldx, const float* logits, int64_t T, int64_t K, int E, int k,
              const float* gs_x, float* gs_out, int32_t* ids, float* w, int32_t* offsets, int32_t* p2f,
              int32_t* f2p, uint8_t* a_codes, uint8_t* a_sf, void* ws, size_t ws_bytes, cudaStream_t s);

// Byte offset of the scale of (row r, 16-element block b) in the tiled layout
// documented in nvfp4moe.h.
// It is the sum of a row part and a block part (c4 = column groups of 64).
__host__ __device__ inline int64_t sf_tiled_row_part(int64_t r, int64_t c4) {
  return (r >> 7) * c4 * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4;
}
__host__ __device__ inline int64_t sf_tiled_block_part(int64_t b) { return (b >> 2) * 512 + (b & 3); }
__host__ __device__ inline int64_t sf_tiled_offset(int64_t r, int64_t b, int64_t c4) {
  return sf_tiled_row_part(r, c4) + sf_tiled_block_part(b);
}

// The same for NVFP4_SF_TILED_ROWS, the layout of the GEMMs' activation (A)
// scales: tiles of 128 rows x 16 blocks (2048 bytes), row-major inside; s =
// ceil(cols / 256) tiles per 128 rows.
__host__ __device__ inline int64_t sf_rows_row_part(int64_t r, int64_t s) { return (r >> 7) * s * 2048 + (r & 127) * 16; }
__host__ __device__ inline int64_t sf_rows_block_part(int64_t b) { return (b >> 4) * 2048 + (b & 15); }
__host__ __device__ inline int64_t sf_rows_offset(int64_t r, int64_t b, int64_t s) {
  return sf_rows_row_part(r, s) + sf_rows_block_part(b);
}

// ------------------------------------------------------------------ NVFP4 encode

// Exact value of an E4M3 byte (every E4M3 value is representable in f16).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
  return __half2float(__half(h));
}

// Round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float v) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// Eight E2M1 codes in one word: q[2j] in the low nibble and q[2j+1] in the
// high nibble of byte j; round to nearest even with saturation at 6. The
// conversion keeps the sign of its input in every case, zeros included
// (checked on sm_103a for -0, negative values that round to 0, negative
// subnormals: all give 0x8), so a negative value that rounds to magnitude 0
// is encoded as 0x8.
__device__ __forceinline__ uint32_t e2m1x8(const float (&q)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return r;
}

// RN(a / s) for an E4M3 block scale s > 0, given rcp = RN(1 / s): the product
// with the reciprocal, corrected by one FMA on its exact remainder. This is the
// final correction step of P. Markstein's FMA-based division ("Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990; also "IA-64 and Elementary Functions", 2000): with an
// exact remainder r = a - q0*s (one FMA) the corrected q0 + r*rcp rounds to the
// correctly rounded quotient. Equal to that quotient bit for bit for every f32
// a and every E4M3 s (checked exhaustively on the host,
// tests/fma_division_check.c); the sign is copied from a so that a = -0 gives -0.
__device__ __forceinline__ float div_by_scale(float a, float s, float rcp) {
  const float q0 = __fmul_rn(a, rcp);
  const float r = __fmaf_rn(-q0, s, a);
  return copysignf(__fmaf_rn(r, rcp, q0), a);
}

// One 16-element block (README "Correctness Bugs Fixed", bugs 3 and 4):
// p = amax * gs; zero or underflowing (p < 6 * 2^-9) blocks get scale 0 and
// codes 0; otherwise sf = E4M3(p / 6) and code_i = E2M1((v_i * gs) / s).
// Every step is a single correctly rounded f32 operation (no contraction); the
// quotient is formed by div_by_scale, which is the correctly rounded one.
// Returns the scale byte; the 16 codes go to w0 (elements 0-7) and w1 (8-15),
// element 2j in the low nibble of byte j.
__device__ __forceinline__ uint32_t quantize_block16(const float (&v)[16], float gs, uint32_t& w0,
                                                     uint32_t& w1) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const float p = __fmul_rn(amax, gs);
  if (!(amax > 0.0f) || p < 0.01171875f) {
    w0 = 0u;
    w1 = 0u;
    return 0u;
  }
  // p / 6 by the same FMA-corrected product (6 is an E4M3 value, so the
  // exhaustive check covers it; p >= 6 * 2^-9 keeps everything normal). From
  // p = 2688 on the scale saturates at 448 whatever the rounding; a plain
  // division there keeps even an infinite p exact.
  const float p6 = p < 2688.0f ? div_by_scale(p, 6.0f, 0x1.555556p-3f) : __fdiv_rn(p, 6.0f);
  const uint32_t sf = f32_to_e4m3_satfinite(p6);
  const float s = e4m3_to_f32(sf);
  const float rcp = __frcp_rn(s);
  float qa[8], qb[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    qa[i] = div_by_scale(__fmul_rn(v[i], gs), s, rcp);
    qb[i] = div_by_scale(__fmul_rn(v[8 + i], gs), s, rcp);
  }
  w0 = e2m1x8(qa);
  w1 = e2m1x8(qb);
  return sf;
}

// Global scale from the bit pattern of a non-negative f32 amax.
__device__ __forceinline__ float global_scale_from_amax_bits(uint32_t bits) {
  const float amax = __uint_as_float(bits);
  return amax > 0.0f ? __fdiv_rn(2688.0f, amax) : 1.0f;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Router step for one token, one warp ("MoE Runner" step 1 input: top-k of
// the router logits, softmax over the k selected). Each lane holds VPL logits
// (expert lane + 32*i); ties go to the lower expert index; the k winners are
// in descending order. Lane j < k receives winner j's expert and weight.
template <int VPL>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k, int lane,
                                            int& my_i, float& my_w) {
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : -INFINITY;
    if (v[i] != v[i]) v[i] = -INFINITY;  // a NaN logit is never preferred (and never leaves no choice)
  }
  uint32_t taken = 0;
  float my_v = -INFINITY;
  my_i = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_v = bv;
      my_i = bi;
    }
  }
  // softmax over the k selected logits; the first selected is the maximum
  const float vmax = __shfl_sync(0xFFFFFFFFu, my_v, 0);
  const float ex = lane < k ? expf(my_v - vmax) : 0.0f;
  float den = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, o);
  my_w = ex / den;
}

// Quantize the 16 BF16 elements at x_row[col0 .. col0+15] (zeros when x_row
// is null); returns the scale byte, the codes in w0/w1.
__device__ __forceinline__ uint32_t quantize_lane16(const __nv_bfloat16* x_row, int64_t col0, float gs,
                                                    uint32_t& w0, uint32_t& w1) {
  float v[16];
  if (x_row) {
    const uint4* p = reinterpret_cast<const uint4*>(x_row + col0);
    bf16x8_to_f32(__ldg(p), v);
    bf16x8_to_f32(__ldg(p + 1), v + 8);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
  }
  return quantize_block16(v, gs, w0, w1);
}

// The scale bytes of lanes 4q..4q+3 as one little-endian word (valid in lane 4q).
__device__ __forceinline__ uint32_t gather_sf_word(uint32_t sf) {
  const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, sf, 1);
  const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, sf, 2);
  const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, sf, 3);
  return sf | (b1 << 8) | (b2 << 16) | (b3 << 24);
}

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 32-byte global store (one full sector); the address is 32-byte aligned.
__device__ __forceinline__ void st_global_32B(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0), "r"(a1), "r"(a2),
               "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

// The same, marked as streaming (written once, read once much later: evicted first).
__device__ __forceinline__ void st_global_32B_stream(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                     uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0), "r"(a1), "r"(a2),
               "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

// 8-byte global store marked as streaming (evict first).
__device__ __forceinline__ void st_global_8B_stream(void* p, uint32_t a0, uint32_t a1) {
  asm volatile("st.global.cs.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(a0), "r"(a1) : "memory");
}

// 16-byte asynchronous copy global -> shared through the load path (L2 only),
// and an arrive on an mbarrier once all of this thread's earlier such copies
// have landed (the barrier's count includes this arrival).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 2-D tiled TMA load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// The same for a CTA of a 2-SM pair: the tile lands in this CTA's shared
// memory and its bytes complete on `bar`, a shared::cluster address that may
// name the mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// tcgen05 (5th-generation tensor core, tensor memory)
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// D (TMEM, f32) (+)= A * B^T with both operands NVFP4 (E2M1 + UE4M3 scale per
// 16 elements along K), M=128, K=64 per instruction.
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}

// Register -> TMEM stores of this warp's 32 lanes (its own lane quadrant):
// one column, or eight consecutive columns.
// Store 1 / 32 consecutive 32-bit columns of this warp's TMEM lane quadrant
// (a store of n columns starts on a column that is a multiple of n).
__device__ __forceinline__ void tc_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
               :: "r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
               : "memory");
}

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 64 consecutive 32-bit columns of this thread's TMEM lane; the registers are
// valid only after tc_wait_ld().
__device__ __forceinline__ void tc_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 64 consecutive 32-bit columns of this thread's TMEM lane, waited for.
__device__ __forceinline__ void tc_ld64_wait(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// ---- thread-block clusters of two CTAs (the 2-SM MMA pairs)

// Rank of this CTA in its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs: arrive (release) and wait (acquire) on the
// cluster's hardware barrier.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address in the shared::cluster window of the variable at shared::cta
// address `addr` in the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive (release at cluster scope) on an mbarrier of another CTA of the
// cluster, given its shared::cluster address.
__device__ __forceinline__ void mbar_remote_arrive(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// The same with relaxed ordering: no release fence, so it costs the issuing
// thread almost nothing (a release at cluster scope measured ~0.4 us per
// arrive). Used where what the arrive announces was already observed complete
// through a local barrier (copies landed, tensor-memory stores or loads waited
// for), so there is nothing left for a release to order.
__device__ __forceinline__ void mbar_remote_arrive_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Store a 32-bit word into another CTA's shared memory (shared::cluster address).
__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Parity wait with acquire at cluster scope (for barriers a peer CTA arrives on).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Tensor memory of a CTA pair: one warp of EACH of the two CTAs executes the
// allocation (and later the deallocation); both receive the same address.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Arrive on the mbarrier at the same shared-memory offset in every CTA of
// `cta_mask` once the pair MMAs this thread issued so far are done.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// The same, on this CTA's own mbarrier only.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// The 2-SM form of tc_mma_nvf4, issued by one thread of the pair's even CTA:
// M = 256 rows, the first 128 from the even CTA's shared memory and the other
// 128 from the odd CTA's (same offsets), N split the same way for B; each CTA
// receives its 128 rows of D in its own tensor memory, and each reads its own
// A scales and the B scales from its own tensor memory.
__device__ __forceinline__ void tc_mma_nvf4_pair(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored as rows of
// 128 bytes with the 128-byte swizzle (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::mxf4nvf4, A and B E2M1 K-major, UE4M3 scales,
// f32 accumulate, shape M x N.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7)                                  // A format: E2M1
         | (1u << 10)                               // B format: E2M1
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (0u << 23)                               // scale format: UE4M3
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

}  // namespace nvfp4moe
