// gdr_walk.cu -- inter-chunk state walk with the chunk outputs, the whole
// 128 x 128 state of one (document, value head) chain in one CTA.
//
// The FP32 state is kept TRANSPOSED in tensor memory: TMEM lane v holds row v
// of S^T (value column v of S), its 128 columns the channels c.  Laid out that
// way the state is directly the A operand of the products that read it
// (tcgen05.mma with A in tensor memory), so no copy of the state ever goes
// through shared memory:
//   [P^T | O^T]  = S0'^T [w ; Qp]^T           (M = 128 value rows, N = 128, K = 128 channels)
//   [O^T | S^T] += Delta^T [Aqk ; Kd^T]^T     (M = 128, N = 192, K = 64 tokens)
// with S0' the state rounded to TF32 (a second TMEM copy, the operand), the
// accumulator P^T pre-loaded with -u^T (so the product leaves u^T - P^T =
// Delta^T ... negated), O^T pre-zeroed, and S^T scaled by diag(gamma) in TMEM
// before the second product.  Per chunk (the chunked identities in
// gdr_common.cuh):
//   Delta = u - w S0,   O = scale (Qp S0 + Aqk Delta),
//   S_end = diag(gamma) S0 + Kd^T Delta.
// The "state walk" and "output program" of PR #8638 "perf(cake_gdn_kcp): ...
// graph-replay checkpoint recompute hands its tapes to the backward" (opening
// description), fused, with the whole value width of a chain on one SM.
//
// Tensor-memory columns (512): Pd[0] 0..63, O[0] 64..127, S 128..255,
// O[1] 256..319, Pd[1] 320..383, S' 384..511.  Chunk m uses Pd[m&1] (P, then
// Delta in place) and O[m&1]: the first product writes [Pd[0] | O[0]] (even m,
// B rows [w ; Qp]) or [O[1] | Pd[1]] (odd m, B rows [Qp ; w]); the second
// accumulates into [O[0] | S] (even, B rows [Aqk ; Kd^T]) or [S | O[1]] (odd,
// B rows [Kd^T ; Aqk]).  The other parity's buffers are drained and refilled
// off the chunk-to-chunk chain.
//
// Threads: 8 data warps (warp w: TMEM lanes 32 (w % 4) .., value rows v; warp
// halves w / 4 split the columns) and one issuer warp (its lane 0 issues every
// TMA copy and MMA).  Shared memory holds the B operands only, two stages
// each: [w ; Qp] (64 KB) and [Kd^T ; Aqk] + gamma (48 KB).  Waits are bounded;
// a timed-out wait ends the walk for the whole CTA and sets the device error
// word.
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "gdr_tc.cuh"

namespace gdr {

struct WalkVSmem {
  float B1[2][2 * CH * DK];       // per stage: 4 column blocks of 128 rows x 32 (16 KB each)
  float B2[2][(DK + CH) * CH];    // per stage: 2 column blocks of 192 rows x 32 (24 KB each)
  float gam[2][DK];               // gamma, with the B2 stage
  uint64_t bar_b1[2], bar_b2[2], bar_s1, bar_s2;
  uint32_t tmem;
};
constexpr int WALKV_THREADS = 288;
constexpr uint32_t WALKV_B1_BYTES = 2 * CH * DK * 4;
constexpr uint32_t WALKV_B2_BYTES = (DK + CH) * CH * 4 + DK * 4;
constexpr uint32_t kColS = 128, kColSp = 384;
__device__ __forceinline__ uint32_t colPd(int b) { return b ? 320u : 0u; }   // P, then Delta, of parity b
__device__ __forceinline__ uint32_t colO(int b) { return b ? 256u : 64u; }   // O of parity b
__device__ __forceinline__ uint32_t colD1(int b) { return b ? 256u : 0u; }   // D of [P | O] / [O | P]
__device__ __forceinline__ uint32_t colD2(int b) { return b ? 128u : 64u; }  // D of [O | S] / [S | O]

__global__ void __launch_bounds__(WALKV_THREADS, 1) k_walk_fwd_v(const __grid_constant__ WalkArgs a) {
  extern __shared__ unsigned char smraw[];
  WalkVSmem& s = *reinterpret_cast<WalkVSmem*>(tc::align1024(smraw));
  const int rank = a.rank_base + blockIdx.x / a.HV;  // all heads of the longest document first
  const int h = blockIdx.x % a.HV;
  const int doc = a.order[rank];
  const DocDesc dd = a.docs[doc];
  const int n = dd.nchunks;
  const int tid = threadIdx.x, warp = tid >> 5, lane = lane_id();
  const bool data = tid < 256, issuer = tid == 256;
  const int q4 = warp & 3, hf = (warp >> 2) & 1;
  const int v = 32 * q4 + lane;  // value row of a data thread
  const size_t sidx = ((size_t)doc * a.HV + h) * DK * DK;

  if (issuer) {
    tc::mbar_init(&s.bar_b1[0], 1);
    tc::mbar_init(&s.bar_b1[1], 1);
    tc::mbar_init(&s.bar_b2[0], 1);
    tc::mbar_init(&s.bar_b2[1], 1);
    tc::mbar_init(&s.bar_s1, 1);
    tc::mbar_init(&s.bar_s2, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&s.tmem, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = s.tmem;
  const uint32_t tl = tm + ((uint32_t)(32 * q4) << 16);  // this warp's lanes

  // Issuer only.  Stage b = m & 1 of each operand.
  auto issue_b1 = [&](int m) {  // [w ; Qp] (even) or [Qp ; w] (odd)
    const int b = m & 1, item = (dd.chunk0 + m) * a.HV + h;
    unsigned char* base = reinterpret_cast<unsigned char*>(s.B1[b]);
    const int wr = b ? 64 : 0, qr = b ? 0 : 64;
    tc::mbar_arrive_expect_tx(&s.bar_b1[b], WALKV_B1_BYTES);
    for (int kb = 0; kb < 4; ++kb) {
      tc::tma_load_2d(base + kb * 16384 + wr * 128, &a.w_map, kb * 32, item * CH, &s.bar_b1[b]);
      tc::tma_load_2d(base + kb * 16384 + qr * 128, &a.qp_map, kb * 32, item * CH, &s.bar_b1[b]);
    }
  };
  auto issue_b2 = [&](int m) {  // [Aqk ; Kd^T] (even) or [Kd^T ; Aqk] (odd), and gamma
    const int b = m & 1, item = (dd.chunk0 + m) * a.HV + h;
    unsigned char* base = reinterpret_cast<unsigned char*>(s.B2[b]);
    const int ar = b ? 128 : 0, kr = b ? 0 : 64;
    tc::mbar_arrive_expect_tx(&s.bar_b2[b], WALKV_B2_BYTES);
    for (int kb = 0; kb < 2; ++kb) {
      tc::tma_load_2d(base + kb * 24576 + ar * 128, &a.aqk_map, kb * 32, item * CH, &s.bar_b2[b]);
      tc::tma_load_2d(base + kb * 24576 + kr * 128, &a.kdt_map, kb * 32, item * DK, &s.bar_b2[b]);
    }
    tc::bulk_load(s.gam[b], &a.gam[(size_t)item * DK], DK * 4, &s.bar_b2[b]);
  };
  // u of chunk m, rows j = 32 hf .. 32 hf + 31 at value column v, negated,
  // into the P accumulator Pd[m & 1] (data threads).
  auto load_neg_u = [&](int m) {
    const float* up = a.u + tf_off(dd.chunk0 + m, h, a.HV) + (size_t)(32 * hf) * LDF + v;
    uint32_t r[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(-__ldg(up + (size_t)j * LDF));
    tc::tmem_st32(tl + colPd(m & 1) + 32 * hf, r);
  };
  // scale * O of chunk m (buffer O[m & 1]) -> out; the buffer is zeroed again
  // for chunk m + 2 (data threads).
  auto drain_out = [&](int m) {
    const int i0 = 32 * hf, len = min(CH, dd.len - CH * m);
    uint32_t r[32];
    tc::tmem_ld32(tl + colO(m & 1) + i0, r);
    tc::tmem_wait_ld();
    __nv_bfloat16* op = a.out + ((size_t)(dd.tok0 + CH * m + i0) * a.HV + h) * DK + v;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i0 + i < len) op[(size_t)i * a.HV * DK] = __float2bfloat16_rn(a.scale * __uint_as_float(r[i]));
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = 0u;
    tc::tmem_st32(tl + colO(m & 1) + i0, r);
  };

  if (data) {
    // S <- h0 (or 0), transposed: S^T[v][c] = h0[c][v].
    uint32_t r[32];
#pragma unroll
    for (int cb = 0; cb < 64; cb += 32) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int c = 64 * hf + cb + j;
        r[j] = __float_as_uint(a.h0 ? a.h0[sidx + (size_t)c * DK + v] : 0.f);
      }
      tc::tmem_st32(tl + kColS + 64 * hf + cb, r);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = 0u;
    tc::tmem_st32(tl + colO(0) + 32 * hf, r);
    tc::tmem_st32(tl + colO(1) + 32 * hf, r);
    if (n > 0) load_neg_u(0);
    tc::tmem_wait_st();
  }
  // Copies issued and consumed (issuer), for the drain after a timeout.
  int b1_iss[2] = {0, 0}, b1_got[2] = {0, 0}, b2_iss[2] = {0, 0}, b2_got[2] = {0, 0}, s1_iss = 0, s2_iss = 0;
  if (issuer) {
    for (int m = 0; m < 2 && m < n; ++m) {
      issue_b1(m), ++b1_iss[m];
      issue_b2(m), ++b2_iss[m];
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();

  constexpr uint32_t kId1 = tc::idesc_tf32(128, 128), kId2 = tc::idesc_tf32(128, 192);
  bool ok = true;
  int m = 0;
  for (; m < n; ++m) {
    const int b = m & 1;
    const int chunk = dd.chunk0 + m;
    uint32_t s0[64];  // S0 row v, columns 64 hf .. 64 hf + 63 (data threads)
    if (data) {
      if (m > 0) {
        ok = tc::mbar_wait(&s.bar_s2, (m - 1) & 1) && ok;  // S0 of this chunk, O of the previous one
        tc::tc_fence_after();
      }
      tc::tmem_ld32(tl + kColS + 64 * hf, s0);
      tc::tmem_ld32(tl + kColS + 64 * hf + 32, s0 + 32);
      tc::tmem_wait_ld();
      uint32_t r[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = tf32(__uint_as_float(s0[32 * half + j]));
        tc::tmem_st32(tl + kColSp + 64 * hf + 32 * half, r);
      }
      tc::tmem_wait_st();
    }
    tc::tc_fence_before();
    if (!named_sync_and(1, WALKV_THREADS, ok)) break;  // S0' is in place
    tc::tc_fence_after();
    if (issuer) {
      const bool r1 = tc::mbar_wait(&s.bar_b1[b], b1_got[b] & 1);
      ok = r1 && ok;
      if (r1) {
        ++b1_got[b];
        tc::tc_fence_after();
        const uint64_t bd = tc::desc_k_sw128(s.B1[b]);
#pragma unroll
        for (int k = 0; k < DK / 8; ++k) tc::mma_tf32_ta(tm + colD1(b), tm + kColSp + 8 * k, tc::kstep32(bd, k, 128), kId1, 1);
        tc::mma_commit(&s.bar_s1);
        ++s1_iss;
      }
    }
    if (data) {
      // While [P | O] runs: diag(gamma) S0 into S, the tape row, the previous
      // chunk's output, -u of the next chunk.
      const bool rg = tc::mbar_wait(&s.bar_b2[b], (m >> 1) & 1);  // gamma of this chunk
      ok = rg && ok;
      const float* gm = s.gam[b] + 64 * hf;
      uint32_t r[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(s0[32 * half + j]) * gm[32 * half + j]);
        tc::tmem_st32(tl + kColS + 64 * hf + 32 * half, r);
      }
      if (a.tape) {  // S0[c][v] as BF16
        __nv_bfloat16* tp = a.tape + state_off(chunk, h, a.HV) + (size_t)(64 * hf) * DK + v;
#pragma unroll
        for (int j = 0; j < 64; ++j) tp[(size_t)j * DK] = __float2bfloat16_rn(__uint_as_float(s0[j]));
      }
      if (m > 0) drain_out(m - 1);
      if (m + 1 < n) load_neg_u(m + 1);
      tc::tmem_wait_st();
      // Delta = -(P - u), rounded to TF32 in place (the A operand of the
      // second product); the FP32 Delta for the backward.
      ok = tc::mbar_wait(&s.bar_s1, m & 1) && ok;
      tc::tc_fence_after();
      tc::tmem_ld32(tl + colPd(b) + 32 * hf, r);
      tc::tmem_wait_ld();
      float* dp = a.delta ? a.delta + tile_off(chunk, h, a.HV) + (size_t)(32 * hf) * DK + v : nullptr;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float d = -__uint_as_float(r[j]);
        if (dp) dp[(size_t)j * DK] = d;
        r[j] = tf32(d);
      }
      tc::tmem_st32(tl + colPd(b) + 32 * hf, r);
      tc::tmem_wait_st();
    }
    tc::tc_fence_before();
    if (!named_sync_and(2, WALKV_THREADS, ok)) break;  // Delta, gamma S0 in place
    tc::tc_fence_after();
    if (issuer) {
      const bool r2 = tc::mbar_wait(&s.bar_b2[b], b2_got[b] & 1);
      ok = r2 && ok;
      if (r2) {
        ++b2_got[b];
        tc::tc_fence_after();
        const uint64_t bd = tc::desc_k_sw128(s.B2[b]);
#pragma unroll
        for (int k = 0; k < CH / 8; ++k) tc::mma_tf32_ta(tm + colD2(b), tm + colPd(b) + 8 * k, tc::kstep32(bd, k, 192), kId2, 1);
        tc::mma_commit(&s.bar_s2);
        ++s2_iss;
      }
      // [P | O] of this chunk is done (the data threads waited for it): its
      // B1 stage takes chunk m + 2.  The B2 stage once the update is done.
      if (ok && m + 2 < n) issue_b1(m + 2), ++b1_iss[b];
      if (ok && m + 2 < n) {
        const bool r3 = tc::mbar_wait(&s.bar_s2, m & 1);
        ok = r3 && ok;
        if (r3) issue_b2(m + 2), ++b2_iss[b];
      }
    }
  }
  if (m < n) {
    // A wait ran out: record it and drain the copies and products in flight.
    if (issuer) {
      atomicExch(a.err, 3);
      for (int q = 0; q < 2; ++q) {
        if (b1_iss[q] > b1_got[q]) tc::mbar_wait(&s.bar_b1[q], (b1_iss[q] - 1) & 1);
        if (b2_iss[q] > b2_got[q]) tc::mbar_wait(&s.bar_b2[q], (b2_iss[q] - 1) & 1);
      }
      if (s1_iss > 0) tc::mbar_wait(&s.bar_s1, (s1_iss - 1) & 1);
      if (s2_iss > 0) tc::mbar_wait(&s.bar_s2, (s2_iss - 1) & 1);
    }
  } else if (data) {
    if (n > 0) {
      ok = tc::mbar_wait(&s.bar_s2, (n - 1) & 1) && ok;
      tc::tc_fence_after();
      if (ok) drain_out(n - 1);
    }
    if (a.ht && ok) {  // ht[c][v] = S^T[v][c]
      uint32_t r[32];
#pragma unroll
      for (int cb = 0; cb < 64; cb += 32) {
        tc::tmem_ld32(tl + kColS + 64 * hf + cb, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) a.ht[sidx + (size_t)(64 * hf + cb + j) * DK + v] = __uint_as_float(r[j]);
      }
    }
    if (!ok) atomicExch(a.err, 3);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tm, 512);
}

cudaError_t launch_walk_fwd_v(const WalkArgs& a, int ndocs, cudaStream_t st) {
  if (ndocs == 0) return cudaSuccess;
  const size_t sm = sizeof(WalkVSmem) + 1024;
  cudaFuncSetAttribute(k_walk_fwd_v, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  k_walk_fwd_v<<<ndocs * a.HV, WALKV_THREADS, sm, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdr
