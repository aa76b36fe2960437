// gdr_common.cuh -- shared device helpers for the chunked gated delta rule.
//
// Chunked form (chunk C = 64 tokens, head dim 128), per (document, value head)
// chain, derived from the token recurrence
//   S_t = (I - beta_t k_t k_t^T) diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
//   o_t = scale * S_t^T q_t
// (the method of flashinfer PR #8218 "feat(cake_kda): ... Cake KDA
// context-parallel (KCP) autograd backend" and PR #7723 "perf(cake_gdn):
// prefetch offset adjoint walk, default LPT segment plan").  Inside one chunk
// with start state S0, chunk-local cumulative log-decay gc_i = sum_{j<=i} g_j,
// Gamma_i = exp(gc_i), gamma = Gamma_last:
//   At  = strict_tril( (K*Gamma) (K/Gamma)^T )    (never formed that way: see
//   Aqk = tril( (Q*Gamma) (K/Gamma)^T )             the block factorization)
//   T   = (I + diag(beta) At)^-1
//   w   = T diag(beta) (K*Gamma),   u = T diag(beta) V
//   Delta = u - w S0
//   O   = scale ( (Q*Gamma) S0 + Aqk Delta )
//   S_end = diag(gamma) S0 + Kd^T Delta,   Kd = K * exp(gc_last - gc)
//
// Per-channel decays exp(gc_i - gc_j) are never split as exp(gc_i)*exp(-gc_j)
// over a whole chunk (exp(-gc) overflows FP32 after ~18 tokens at g = -5).
// Instead products over channels are factored per 16-row block with the
// reference point r = gc at the block's 8th row: for rows i of the block and
// columns j <= i, exp(gc_i - gc_j) = exp(gc_i - r) * exp(r - gc_j), where the
// row factor lies within exp(+-8 max|g|) (2^+-116 for g >= -10, finite in FP32)
// and the column factor is <= 1 for every j before the 8th row and within
// exp(8 max|g|) after it.  A column factor that flushes to zero belongs to a
// term below 2^-25 of the result.
//
// Matrix products use warp-level mma.sync m16n8k8 with TF32 operands
// (round-to-nearest) and FP32 accumulation.  BF16 operands were measured on
// the CPU emulation to miss the output tolerance; TF32 does not.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gdr {

constexpr int CH = 64;     // chunk length (tokens)
constexpr int DK = 128;    // head dimension (K = V = 128)
constexpr int LDT = 132;   // shared-memory row stride of a [64][128] FP32 tile
constexpr int LDS = 68;    // shared-memory row stride of a [64][64] FP32 tile
constexpr int LDF = 136;   // [64][128] FP32 tile stride for reads with the row on the thread-in-group index
constexpr float LOG2E = 1.4426950408889634f;

// One 64-token chunk of one document.  Chunks restart at every document start.
struct ChunkDesc {
  int tok0;   // first token (index into the packed T axis)
  int len;    // 1..64 valid rows
  int doc;    // document index
  int idx;    // chunk index within the document
};

// One document: its token range and its chunks [chunk0, chunk0 + nchunks).
struct DocDesc {
  int tok0, len, chunk0, nchunks;
};

// One segment of a document's chunks, the unit of work of a state-walk CTA.
// A document of n chunks is split into nseg >= 1 segments of balanced length
// (the first n % nseg get one chunk more); an empty document is one empty
// segment.  Segments are numbered in the walks' document order, so that the
// segments of a run of documents form one contiguous range.
struct SegDesc {
  int doc;      // document index
  int tok0;     // first token
  int len;      // tokens
  int chunk0;   // first chunk (global chunk index)
  int nchunks;  // chunks
  int idx;      // index within the document
  int nseg;     // segments of the document
  int first;    // global index of the document's first segment
};

// An MMA operand at TF32 precision, rounded to nearest with ties away from
// zero: half a unit in the last TF32 place is added to the magnitude bits (a
// carry into the exponent is the correct rounding up).  The tensor cores read
// a TF32 operand's 19 high bits (sign, exponent, 10 mantissa bits) and ignore
// the 13 low bits left behind; tf32_value clears them, for code that uses the
// rounded number itself.  One integer add per element.
__device__ __forceinline__ uint32_t tf32(float x) { return __float_as_uint(x) + 0x1000u; }
__device__ __forceinline__ uint32_t tf32_value(float x) { return (__float_as_uint(x) + 0x1000u) & 0xffffe000u; }

// 2^x (the PTX approximate base-2 exponential).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// D += A * B, m16n8k8, TF32 inputs, FP32 accumulate.
__device__ __forceinline__ void mma8(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// d += a b with FP32 operands split as x = hi + lo (hi = x rounded to TF32,
// lo = the remainder rounded to TF32): about FP32 accuracy from three TF32
// products, lo*hi, hi*lo and hi*hi, each into an accumulator of its own
// (d[0], d[1], d[2]: three independent chains instead of one three times as
// long); the caller adds them, small terms first, as (d[0] + d[1]) + d[2].
__device__ __forceinline__ void mma8_split3(float (&d)[3][4], const float (&a)[4], const float (&b)[2]) {
  uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ah[i] = tf32_value(a[i]);
    al[i] = tf32(a[i] - __uint_as_float(ah[i]));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    bh[i] = tf32_value(b[i]);
    bl[i] = tf32(b[i] - __uint_as_float(bh[i]));
  }
  mma8(d[0], al, bh);
  mma8(d[1], ah, bl);
  mma8(d[2], ah, bh);
}


// 16-byte asynchronous global -> shared copy (L2 only) and its group fences.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ float bfbits2f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Four 8x8 matrices of 16-bit elements from shared memory, transposed on the
// way (ldmatrix .trans): lane l gives the address of row l % 8 of matrix l / 8
// (16 contiguous bytes); register m of lane l receives column l / 4 of matrix
// m at rows 2 (l % 4) (low half) and 2 (l % 4) + 1 (high half).
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void* row) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(row));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
// The two BF16 values of a packed pair as FP32 (low half, high half).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Barrier over `count` threads (a multiple of 32) on hardware barrier `id` (1..15).
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// Barrier over `count` threads on hardware barrier `id`; returns true on every
// participating thread iff `pred` was true on all of them.
__device__ __forceinline__ bool named_sync_and(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// Fragment coordinates (PTX m16n8k8 .tf32 layouts):
//   A: a0 (g, t) a1 (g+8, t) a2 (g, t+4) a3 (g+8, t+4)      [row, k]
//   B: b0 (t, g) b1 (t+4, g)                                [k, col]
//   C: c0 (g, 2t) c1 (g, 2t+1) c2 (g+8, 2t) c3 (g+8, 2t+1)  [row, col]
// with g = lane / 4, t = lane % 4.  Which k index fills which of a step's
// eight k slots is free as long as A and B agree, so kernels put adjacent
// elements in slots t and t + 4 where that makes the operand reads pairs or
// conflict-free; with the assignments used here the outputs came out bit for
// bit those of the plain order (compared on whole forward and backward
// passes).

// One k-step of 8 (k0 .. k0+7) of a warp product C[16 x 8*NT] += A * B over
// n-tiles [nt0, nt1).  fa(i, k) and fb(k, n) return FP32 values.
template <int NT, class FA, class FB>
__device__ __forceinline__ void mma_kstep(float (&acc)[NT][4], int k0, int nt0, int nt1, FA fa, FB fb) {
  const int lane = lane_id(), g = lane >> 2, t = lane & 3;
  uint32_t a[4];
  a[0] = tf32(fa(g, k0 + t));
  a[1] = tf32(fa(g + 8, k0 + t));
  a[2] = tf32(fa(g, k0 + t + 4));
  a[3] = tf32(fa(g + 8, k0 + t + 4));
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if (nt < nt0 || nt >= nt1) continue;
    uint32_t b[2];
    b[0] = tf32(fb(k0 + t, nt * 8 + g));
    b[1] = tf32(fb(k0 + t + 4, nt * 8 + g));
    mma8(acc[nt], a, b);
  }
}

template <int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[NT][4]) {
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
}

// Visit every accumulator element: f(row, col, value&) with row in [0,16).
template <int NT, class F>
__device__ __forceinline__ void acc_foreach(float (&acc)[NT][4], F f) {
  const int lane = lane_id(), g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int r = 0; r < 4; ++r) f(g + 8 * (r >> 1), nt * 8 + 2 * t + (r & 1), acc[nt][r]);
  }
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float ldg_bf(const __nv_bfloat16* p) { return __bfloat162float(__ldg(p)); }

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Offsets into the chunk-major intermediate buffers.
__device__ __forceinline__ size_t tile_off(int chunk, int h, int HV) {  // [NC][HV][64][128]
  return ((size_t)chunk * HV + h) * (CH * DK);
}
__device__ __forceinline__ size_t state_off(int chunk, int h, int HV) { // [NC][HV][128][128]
  return ((size_t)chunk * HV + h) * (DK * DK);
}
// The walks' operand tiles, FP16 with dense rows (element offsets): w [64][128],
// Q Gamma [64][128], Kd^T [128][64], Aqk [64][64].  They depend on q, k, g
// and beta only, so their entries are of order one; FP16 keeps the 11-bit
// significand the TF32 products use.
__device__ __forceinline__ size_t w_off(int chunk, int h, int HV) { return ((size_t)chunk * HV + h) * (CH * DK); }
__device__ __forceinline__ size_t qp_off(int chunk, int h, int HV) { return ((size_t)chunk * HV + h) * (CH * DK); }
__device__ __forceinline__ size_t kd_off(int chunk, int h, int HV) { return ((size_t)chunk * HV + h) * (DK * CH); }
__device__ __forceinline__ size_t aqk_off(int chunk, int h, int HV) { return ((size_t)chunk * HV + h) * (CH * CH); }
// Tiles the gradient kernel moves whole keep its pitches too: dw, dDelta
// [64][LDF] and u (FP16) [64][LDF]; At, T, dAqk [64][LDS].
__device__ __forceinline__ size_t tf_off(int chunk, int h, int HV) { return ((size_t)chunk * HV + h) * (CH * LDF); }
__device__ __forceinline__ size_t ts_off(int chunk, int h, int HV) { return ((size_t)chunk * HV + h) * (CH * LDS); }

}  // namespace gdr
