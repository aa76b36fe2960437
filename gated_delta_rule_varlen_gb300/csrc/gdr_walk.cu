// gdr_walk.cu -- the inter-chunk state walks (forward with the chunk outputs,
// and the reverse adjoint walk), the whole 128 x 128 state of one (document,
// value head) chain in one CTA.
//
// Forward.  The FP32 state is kept TRANSPOSED in tensor memory: TMEM lane v
// holds row v of S^T (value column v of S), its 128 columns the channels c.
// Laid out that way the state is directly the A operand of the products that
// read it (tcgen05.mma with A in tensor memory), so no copy of the state goes
// through shared memory:
//   [P^T | O^T]  = S0'^T [w ; Qp]^T           (M = 128 value rows, N = 128, K = 128 channels)
//   [O^T | S^T] += Delta^T [Aqk ; Kd^T]^T     (M = 128, N = 192, K = 64 tokens)
// as tcgen05.mma kind::f16 series: S0' is the state rounded to FP16 (a second
// TMEM copy, two elements per 32-bit column; the FP32 state stays the
// accumulator), the B tiles [w ; Qp] and [Aqk ; Kd^T] are the FP16 tiles the
// prep stored, Delta^T = u^T - P^T is formed in FP32 by the data warps and
// enters the second product as its FP16 copy Delta'^T, and S^T is scaled by
// diag(gamma) in place before it.  FP16 keeps the 11-bit significand of TF32
// (the operands depend on q, k, g, beta or are of the size of the values v).  Per chunk (the chunked identities in
// gdr_common.cuh):
//   Delta = u - w S0,   O = scale (Qp S0 + Aqk Delta),
//   S_end = diag(gamma) S0 + Kd^T Delta.
// The "state walk" and "output program" of PR #8638 "perf(cake_gdn_kcp): ...
// graph-replay checkpoint recompute hands its tapes to the backward" (opening
// description), fused, with the whole value width of a chain on one SM.
//
// Tensor-memory columns (512): Pd[0] 0..63, O[0] 64..127, S 128..255,
// O[1] 256..319, Pd[1] 320..383, S' 384..447 (FP16 pairs), Delta' 448..479
// (FP16 pairs).  Chunk m uses Pd[m&1] (P, then the FP32 Delta in place) and
// O[m&1]: the first product writes [Pd[0] | O[0]] (even m,
// B rows [w ; Qp]) or [O[1] | Pd[1]] (odd m, B rows [Qp ; w]); the second
// accumulates into [O[0] | S] (even, B rows [Aqk ; Kd^T]) or [S | O[1]] (odd,
// B rows [Kd^T ; Aqk]).  O of a chunk is written out while the next chunk's
// first product runs.
//
// The state tape (S0 of every chunk, BF16, for the backward) is stored
// chunk-major: element (v, c) of a chunk's 128 x 128 tile at
// ((c / 8) * 128 + v) * 8 + c % 8, so that the 32 lanes of a warp (32
// consecutive v) store 512 contiguous bytes per 8-channel piece.
//
// Threads: 8 data warps (warp w: TMEM lanes 32 (w % 4) .., value rows v; warp
// halves w / 4 split the columns) and one issuer warp (its lane 0 issues every
// TMA copy and MMA).  Shared memory: [w ; Qp] + gamma in two stages (32 KB
// each), [Kd^T ; Aqk] (24 KB) and u (16 KB) in one.  Waits are bounded; a
// timed-out wait ends the walk for the whole CTA and sets the device error
// word.
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "gdr_tc.cuh"

namespace gdr {

struct WalkVSmem {
  uint16_t B1[2][2 * CH * DK];  // per stage, FP16: 2 column blocks of 128 rows x 64 channels (16 KB each)
  uint16_t B2[(DK + CH) * CH];  // FP16: 1 column block of 192 rows x 64 tokens
  uint16_t U[CH * DK];         // u (FP16): 2 blocks of 64 rows j x 64 value columns (128-byte swizzle)
  float gam[2][DK];            // gamma, with the B1 stage
  uint64_t bar_b1[2], bar_b2, bar_u, bar_s1, bar_s2;
  uint32_t tmem;
};
constexpr int WALKV_THREADS = 288;
constexpr uint32_t WALKV_B1_BYTES = 2 * CH * DK * 2 + DK * 4;
constexpr uint32_t WALKV_B2_BYTES = (DK + CH) * CH * 2;
constexpr uint32_t WALKV_U_BYTES = CH * DK * 2;
constexpr uint32_t kColS = 128, kColSp = 384;  // S (FP32), S' (FP16 pairs)
constexpr uint32_t kColDl = 448;                // Delta' (FP16 pairs)
__device__ __forceinline__ uint32_t colPd(int b) { return b ? 320u : 0u; }   // P, then Delta, of parity b
__device__ __forceinline__ uint32_t colO(int b) { return b ? 256u : 64u; }   // O of parity b
__device__ __forceinline__ uint32_t colD1(int b) { return b ? 256u : 0u; }   // D of [P | O] / [O | P]
__device__ __forceinline__ uint32_t colD2(int b) { return b ? 128u : 64u; }  // D of [O | S] / [S | O]

// Element offset of (v, c) in a chunk-major BF16 state tile.
__device__ __forceinline__ size_t tape_off(int v, int c) { return ((size_t)(c >> 3) * DK + v) * 8 + (c & 7); }

__global__ void __launch_bounds__(WALKV_THREADS, 1) k_walk_fwd_v(const __grid_constant__ WalkArgs a) {
  extern __shared__ unsigned char smraw[];
  WalkVSmem& s = *reinterpret_cast<WalkVSmem*>(tc::align1024(smraw));
  const int seg = a.seg_base + blockIdx.x / a.HV;  // all heads of the longest document's segments first
  const int h = blockIdx.x % a.HV;
  const SegDesc dd = a.segs[seg];
  const int n = dd.nchunks;
  // What this CTA walks: its segment's full walk with the outputs (mode 0);
  // in the summary launch (mode 1), by blockIdx.y: 0 the first segment of a
  // split document from h0, giving the start state of the second; 1 a middle
  // segment from a zero state (its bias); 2 a middle segment from the
  // identity without u (its state map M).
  int kind = 0;
  if (a.mode == 1) {
    kind = 1 + (int)blockIdx.y;
    const bool on = blockIdx.y == 0 ? (dd.idx == 0 && dd.nseg > 1) : (dd.idx >= 1 && dd.idx <= dd.nseg - 2);
    if (!on) return;
  }
  const bool outputs = kind == 0, use_u = kind != 3;
  // The chunks of this launch, [mb, me) of the segment: all of them, or one
  // slice of a pipelined walk (mb even), which starts from the previous
  // slice's end state and leaves its own in the carry buffer.
  if (kind == 0 && a.m0 > 0 && a.m0 >= n) return;
  const int mb = kind == 0 ? min(a.m0, n) : 0, me = kind == 0 ? min(a.m1, n) : n;
  // Start and end states (S[c][v]): h0 / ht of the document, or per-segment
  // buffers [NSEG][HV][128][128].
  auto start_state = [&]() -> const float* {
    const size_t sidx = ((size_t)dd.doc * a.HV + h) * DK * DK, gidx = ((size_t)seg * a.HV + h) * DK * DK;
    if (kind == 0 && mb > 0) return a.carry + gidx;
    return (kind == 0 && dd.idx > 0) ? a.sstart + gidx : (kind <= 1 && a.h0 ? a.h0 + sidx : nullptr);
  };
  auto end_state = [&]() -> float* {
    const size_t sidx = ((size_t)dd.doc * a.HV + h) * DK * DK, gidx = ((size_t)seg * a.HV + h) * DK * DK;
    if (kind == 0 && me < n) return a.carry + gidx;
    return kind == 0   ? (dd.idx == dd.nseg - 1 && a.ht ? a.ht + sidx : nullptr)
           : kind == 1 ? a.sstart + gidx + (size_t)a.HV * DK * DK
           : kind == 2 ? a.sbias + gidx
                       : a.smap + gidx;
  };
  const int tid = threadIdx.x, warp = tid >> 5, lane = lane_id();
  const bool data = tid < 256, issuer = tid == 256;
  const int q4 = warp & 3, hf = (warp >> 2) & 1;
  const int v = 32 * q4 + lane;  // value row of a data thread

  if (issuer) {
    tc::mbar_init(&s.bar_b1[0], 1);
    tc::mbar_init(&s.bar_b1[1], 1);
    tc::mbar_init(&s.bar_b2, 1);
    tc::mbar_init(&s.bar_u, 1);
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

  // Issuer only.
  auto issue_b1 = [&](int m) {  // [w ; Qp] (even m) or [Qp ; w] (odd m), and gamma, into stage m & 1
    const int b = m & 1, item = (dd.chunk0 + m) * a.HV + h;
    unsigned char* base = reinterpret_cast<unsigned char*>(s.B1[b]);
    const int wr = b ? 64 : 0, qr = b ? 0 : 64;
    tc::mbar_arrive_expect_tx(&s.bar_b1[b], WALKV_B1_BYTES);
    for (int kb = 0; kb < 2; ++kb) {
      tc::tma_load_2d(base + kb * 16384 + wr * 128, &a.w_map, kb * 64, item * CH, &s.bar_b1[b]);
      tc::tma_load_2d(base + kb * 16384 + qr * 128, &a.qp_map, kb * 64, item * CH, &s.bar_b1[b]);
    }
    tc::bulk_load(s.gam[b], &a.gam[(size_t)item * DK], DK * 4, &s.bar_b1[b]);
  };
  auto issue_b2 = [&](int m) {  // [Aqk ; Kd^T] (even m) or [Kd^T ; Aqk] (odd m)
    const int item = (dd.chunk0 + m) * a.HV + h;
    unsigned char* base = reinterpret_cast<unsigned char*>(s.B2);
    const int ar = (m & 1) ? 128 : 0, kr = (m & 1) ? 0 : 64;
    tc::mbar_arrive_expect_tx(&s.bar_b2, WALKV_B2_BYTES);
    tc::tma_load_2d(base + ar * 128, &a.aqk_map, 0, item * CH, &s.bar_b2);
    tc::tma_load_2d(base + kr * 128, &a.kdt_map, 0, item * DK, &s.bar_b2);
  };
  auto issue_u = [&](int m) {
    const int item = (dd.chunk0 + m) * a.HV + h;
    tc::mbar_arrive_expect_tx(&s.bar_u, WALKV_U_BYTES);
    for (int vb = 0; vb < 2; ++vb) tc::tma_load_2d(s.U + vb * CH * 64, &a.u_map, vb * 64, item * CH, &s.bar_u);
  };
  // scale * O of chunk m (buffer O[m & 1]) -> out, rows i = 32 hf .. (data threads).
  auto drain_out = [&](int m) {
    const int i0 = 32 * hf, len = min(CH, dd.len - CH * m);
    uint32_t r[32];
    tc::tmem_ld32(tl + colO(m & 1) + i0, r);
    tc::tmem_wait_ld();
    __nv_bfloat16* op = a.out + ((size_t)(dd.tok0 + CH * m + i0) * a.HV + h) * DK + v;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i0 + i < len) op[(size_t)i * a.HV * DK] = __float2bfloat16_rn(a.scale * __uint_as_float(r[i]));
  };

  if (data) {
    // S <- the start state (h0, a merged segment start, the identity or 0),
    // transposed: S^T[v][c] = start[c][v].
    uint32_t r[32];
    const float* start = start_state();
#pragma unroll
    for (int cb = 0; cb < 64; cb += 32) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int c = 64 * hf + cb + j;
        r[j] = __float_as_uint(start ? start[(size_t)c * DK + v] : (kind == 3 && c == v ? 1.f : 0.f));
      }
      tc::tmem_st32(tl + kColS + 64 * hf + cb, r);
    }
    tc::tmem_wait_st();
  }
  // Copies issued and consumed (issuer), for the drain after a timeout.
  int b1_iss[2] = {0, 0}, b1_got[2] = {0, 0}, b2_iss = 0, b2_got = 0, u_iss = 0, u_got = 0, s1_iss = 0, s2_iss = 0;
  if (issuer && me > mb) {
    issue_b1(mb), ++b1_iss[0];
    if (me - mb > 1) issue_b1(mb + 1), ++b1_iss[1];
    issue_b2(mb), ++b2_iss;
    if (use_u) issue_u(mb), ++u_iss;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();

  constexpr uint32_t kId1 = tc::idesc_f16(128, 128), kId2 = tc::idesc_f16(128, 192);
  bool ok = true;
  int m = mb;
  for (; m < me; ++m) {
    const int mm = m - mb;  // barrier phases count from the launch's first chunk
    const int b = m & 1;
    const int chunk = dd.chunk0 + m;
    if (data) {
      if (mm > 0) {
        ok = tc::mbar_wait(&s.bar_s2, (mm - 1) & 1) && ok;  // S0 of this chunk, O of the previous one
        tc::tc_fence_after();
      }
      ok = tc::mbar_wait(&s.bar_b1[b], (mm >> 1) & 1) && ok;  // gamma of this chunk
      // Columns 64 hf .. 64 hf + 63 in two halves: the tape tile (chunk-major: 512
      // contiguous bytes per warp and 8-channel piece), S0' = S0 rounded to FP16
      // (the A operand, two channels per column), and diag(gamma) S0 into S.  (Scaling S while [P | O]
      // runs instead measured slower: the products read their A operand from
      // tensor memory, and the warps' tensor-memory traffic slows them.)
      const float* gm = s.gam[b] + 64 * hf;
      __nv_bfloat16* tp = a.tape && outputs ? a.tape + state_off(chunk, h, a.HV) : nullptr;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int c0 = 64 * hf + 32 * half;
        uint32_t s0[32], r[32];
        tc::tmem_ld32(tl + kColS + c0, s0);
        tc::tmem_wait_ld();
        if (tp) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            __nv_bfloat162 p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              p[e] = __floats2bfloat162_rn(__uint_as_float(s0[8 * q + 2 * e]), __uint_as_float(s0[8 * q + 2 * e + 1]));
            *reinterpret_cast<uint4*>(tp + tape_off(v, c0 + 8 * q)) = *reinterpret_cast<uint4*>(p);
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const __half2 p = __floats2half2_rn(__uint_as_float(s0[2 * j]), __uint_as_float(s0[2 * j + 1]));
          r[j] = *reinterpret_cast<const uint32_t*>(&p);
        }
        tc::tmem_st16(tl + kColSp + c0 / 2, *reinterpret_cast<const uint32_t(*)[16]>(r));
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(s0[j]) * gm[32 * half + j]);
        tc::tmem_st32(tl + kColS + c0, r);
      }
      tc::tmem_wait_st();
    }
    tc::tc_fence_before();
    if (!named_sync_and(1, WALKV_THREADS, ok)) break;  // S0', diag(gamma) S0 in place
    tc::tc_fence_after();
    if (issuer) {
      ok = tc::mbar_wait(&s.bar_b1[b], (mm >> 1) & 1) && ok;  // complete: the data threads waited for it
      ++b1_got[b];
      tc::tc_fence_after();
      const uint64_t bd = tc::desc_k_sw128(s.B1[b]);
#pragma unroll
      for (int k = 0; k < DK / 16; ++k)
        tc::mma_f16_ta(tm + colD1(b), tm + kColSp + 8 * k, tc::kstep32(bd, k, 128), kId1, k > 0);
      tc::mma_commit(&s.bar_s1);
      ++s1_iss;
    }
    if (data) {
      // While [P | O] runs: the previous chunk's output.
      if (outputs && mm > 0) drain_out(m - 1);
      // Delta = u - P (rows j = 32 hf ..) in FP32 in place (for the backward),
      // and its FP16 copy (the A operand of the second product).
      ok = tc::mbar_wait(&s.bar_s1, mm & 1) && ok;
      if (use_u) ok = tc::mbar_wait(&s.bar_u, mm & 1) && ok;
      tc::tc_fence_after();
      uint32_t r[32];
      tc::tmem_ld32(tl + colPd(b) + 32 * hf, r);
      tc::tmem_wait_ld();
      const int vv = v & 63;  // u[j][v]: block v / 64, 16-byte piece vv / 8 (swizzled by j), element vv % 8
      const unsigned char* ub = reinterpret_cast<const unsigned char*>(s.U) + (v >> 6) * (CH * 128) + (vv & 7) * 2;
      uint32_t rr[16];
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int j = 32 * hf + jj;
        const float uu = use_u ? __half2float(*reinterpret_cast<const __half*>(ub + j * 128 + (((vv >> 3) ^ (j & 7)) << 4)))
                               : 0.f;
        r[jj] = __float_as_uint(uu - __uint_as_float(r[jj]));
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const __half2 p = __floats2half2_rn(__uint_as_float(r[2 * q]), __uint_as_float(r[2 * q + 1]));
        rr[q] = *reinterpret_cast<const uint32_t*>(&p);
      }
      tc::tmem_st32(tl + colPd(b) + 32 * hf, r);      // FP32 Delta, written out below
      tc::tmem_st16(tl + kColDl + 16 * hf, rr);       // FP16 Delta, the A operand of the update
      tc::tmem_wait_st();
    }
    tc::tc_fence_before();
    if (!named_sync_and(2, WALKV_THREADS, ok)) break;  // Delta in place; u read
    tc::tc_fence_after();
    if (data && a.delta && outputs) {  // the FP32 Delta for the backward, while the update runs
      uint32_t r[32];
      tc::tmem_ld32(tl + colPd(b) + 32 * hf, r);
      tc::tmem_wait_ld();
      float* dp = a.delta + tile_off(chunk, h, a.HV) + (size_t)(32 * hf) * DK + v;
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) dp[(size_t)jj * DK] = __uint_as_float(r[jj]);
    }
    if (issuer) {
      const bool r2 = tc::mbar_wait(&s.bar_b2, b2_got & 1);
      ok = r2 && ok;
      if (r2) {
        ++b2_got;
        u_got += use_u;
        tc::tc_fence_after();
        const uint64_t bd = tc::desc_k_sw128(s.B2);
#pragma unroll
        for (int k = 0; k < CH / 16; ++k)
          tc::mma_f16_ta(tm + colD2(b), tm + kColDl + 8 * k, tc::kstep32(bd, k, 192), kId2, 1);
        tc::mma_commit(&s.bar_s2);
        ++s2_iss;
      }
      // Refills: stage b of [w ; Qp] (its product is done) with chunk m + 2,
      // u (read before the barrier) and, once the update is done, [Kd^T ;
      // Aqk] with chunk m + 1.
      if (ok && m + 2 < me) issue_b1(m + 2), ++b1_iss[b];
      if (ok && m + 1 < me) {
        if (use_u) issue_u(m + 1), ++u_iss;
        const bool r3 = tc::mbar_wait(&s.bar_s2, mm & 1);
        ok = r3 && ok;
        if (r3) issue_b2(m + 1), ++b2_iss;
      }
    }
  }
  if (m < me) {
    // A wait ran out: record it and drain the copies and products in flight.
    if (issuer) {
      atomicExch(a.err, 3);
      for (int q = 0; q < 2; ++q)
        if (b1_iss[q] > b1_got[q]) tc::mbar_wait(&s.bar_b1[q], (b1_iss[q] - 1) & 1);
      if (b2_iss > b2_got) tc::mbar_wait(&s.bar_b2, (b2_iss - 1) & 1);
      if (u_iss > u_got) tc::mbar_wait(&s.bar_u, (u_iss - 1) & 1);
      if (s1_iss > 0) tc::mbar_wait(&s.bar_s1, (s1_iss - 1) & 1);
      if (s2_iss > 0) tc::mbar_wait(&s.bar_s2, (s2_iss - 1) & 1);
    }
  } else if (data) {
    if (me > mb) {
      ok = tc::mbar_wait(&s.bar_s2, (me - 1 - mb) & 1) && ok;
      tc::tc_fence_after();
      if (ok && outputs) drain_out(me - 1);
    }
    float* end = end_state();
    if (end && ok) {  // end[c][v] = S^T[v][c]
      uint32_t r[32];
#pragma unroll
      for (int cb = 0; cb < 64; cb += 32) {
        tc::tmem_ld32(tl + kColS + 64 * hf + cb, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) end[(size_t)(64 * hf + cb + j) * DK + v] = __uint_as_float(r[j]);
      }
    }
    if (!ok) atomicExch(a.err, 3);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tm, 512);
}

cudaError_t launch_walk_fwd_v(const WalkArgs& a, int nsegs, cudaStream_t st) {
  if (nsegs == 0) return cudaSuccess;
  const size_t sm = sizeof(WalkVSmem) + 1024;
  cudaFuncSetAttribute(k_walk_fwd_v, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  k_walk_fwd_v<<<dim3(nsegs * a.HV, a.mode == 1 ? 3 : 1), WALKV_THREADS, sm, st>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Reverse adjoint walk, the whole 128 x 128 adjoint of one (document, value
// head) chain in one CTA, chunks in reverse.  With dS the adjoint of the
// chunk's end state (the chunked identities in gdr_bwd.cu's header):
//   dDelta = scale Aqk^T dO + Kd dS
//   dS0    = diag(gamma) dS + scale Qp^T dO - w^T dDelta
// The adjoint is kept transposed in tensor memory (lane v, columns c) and is
// the A operand (from tensor memory) of the products that read it:
//   dDelta^T  = dS'^T Kd^T                                (M = 128, N = 64, K = 128 channels)
//   [dDelta^T | dS^T] += (scale dO)'^T [Aqk^T ; Qp^T]^T  (M = 128, N = 192, K = 64 tokens)
//   dS^T += (-dDelta')^T (w^T)^T                          (M = 128, N = 128, K = 64 tokens)
// (primes: TF32-rounded copies in tensor memory; dS^T is scaled by
// diag(gamma) in place before the second product).  The adjoints are
// gradients, whose scale the caller's loss sets, so these products keep
// TF32 operands (FP32 range).  They contract each saved tile over its other
// index than the forward's products do, and TF32 operands must be K-major,
// so the B operands are the forward's tiles transposed: TMA brings each
// chunk's FP16 tiles as stored (w, Q Gamma, Kd^T, Aqk) into a staging area,
// and the data warps transpose them, 4 x 4 elements per thread, into the
// 128-byte-swizzled K-major FP32 operand stage (FP16 values are exact in
// TF32), each tile just before the product that reads it: Kd with the adjoint's copy, [Aqk^T ;
// Qp^T] before the second product, w^T while it runs.  A staging group is
// refilled with the next chunk's tiles as soon as it has been transposed, a
// whole chunk ahead of its next use.  Each chunk stores the adjoint of its
// end state as the BF16 dS tape (chunk-major like the state tape) and dDelta
// (FP32).
// The "adjoint walk" of PR #7723 "perf(cake_gdn): prefetch offset adjoint
// walk, default LPT segment plan" (opening description), which also
// prefetches its operands one step ahead.
//
// Tensor-memory columns: dDelta 0..63, dS 64..191, dS' 192..319, (scale dO)'
// for even and odd steps 320..383 and 384..447, -dDelta' (TF32) 448..511.
// ---------------------------------------------------------------------------
struct WalkBvSmem {
  // Operand stage (K-major, 128-byte swizzle):
  float BA[(CH + DK) * CH];  // [Aqk^T ; Qp^T]: rows j then c, K = i; 2 column blocks of 192 rows
  float BK[CH * DK];         // Kd [j][c]: rows j, K = c; 4 column blocks of 64 rows
  float BW[DK * CH];         // w^T [c][j]: rows c, K = j; 2 column blocks of 128 rows
  // Staging, the saved FP16 tiles as the forward reads them (TMA, 128-byte swizzle):
  uint16_t SK[DK * CH];      // Kd^T [c][j]: 1 column block of 128 rows
  uint16_t SA[CH * CH];      // Aqk [i][j]: 1 column block of 64 rows
  uint16_t SQ[CH * DK];      // Q Gamma [i][c]: 2 column blocks of 64 rows
  uint16_t SW[CH * DK];      // w [j][c]: 2 column blocks of 64 rows
  float gam[DK];             // gamma, with the Kd^T group
  uint64_t bar_k, bar_a, bar_w, bar_ab, bar_c;
  uint32_t tmem;
};
constexpr uint32_t kBColD = 0, kBColS = 64, kBColSp = 192, kBColDn = 448;
__device__ __forceinline__ uint32_t colDO(int b) { return b ? 384u : 320u; }
constexpr uint32_t WALKB_K_BYTES = DK * CH * 2 + DK * 4, WALKB_A_BYTES = (CH * CH + CH * DK) * 2,
                   WALKB_W_BYTES = CH * DK * 2;

// Byte offset of FP32 element (row r, k) of a K-major 128B-swizzled operand of
// R rows (column blocks of 32 k).
__device__ __forceinline__ uint32_t sw_off(int r, int k, int R) {
  return (uint32_t)((k >> 5) * R * 128 + r * 128 + ((((k & 31) >> 2) ^ (r & 7)) << 4) + ((k & 3) << 2));
}

// Byte offset of FP16 element (row r, k) of a 128B-swizzled tile of R rows
// (column blocks of 64 k).
__device__ __forceinline__ uint32_t sw_off_h(int r, int k, int R) {
  return (uint32_t)((k >> 6) * R * 128 + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4) + ((k & 7) << 1));
}

// One group of 32 4 x 4 blocks of a transposed copy from a 128B-swizzled FP16
// tile to a K-major 128B-swizzled FP32 tile: source rows sr0 .. sr0+15 (of
// R_s rows), source columns sc0 .. sc0+31 become destination rows roff + sc0
// .. (of R_d rows) with the source rows as their K index.  A 16-byte shared access is served a quarter
// warp at a time, so the eight lanes of each quarter take row quads and column
// quads such that their reads (row 4 rq + a, column chunk cq) and their writes
// (row 4 cq + b, K chunk rq) each fall on eight different 16-byte bank groups:
// lane (quarter qq, index i) takes row quad 2 ((i >> 1) & 1) + (i >> 2) and
// column quad (i & 1) + 2 (((i >> 1) & 1) ^ (qq & 1)) + 4 (qq >> 1).
__device__ __forceinline__ void transpose_group(const unsigned char* src, int Rs, int sr0, int sc0, unsigned char* dst,
                                                int Rd, int roff) {
  const int l = lane_id(), qq = l >> 3, i = l & 7;
  const int rq = 2 * ((i >> 1) & 1) + (i >> 2), cq = (i & 1) + 2 * (((i >> 1) & 1) ^ (qq & 1)) + 4 * (qq >> 1);
  const int r0 = sr0 + 4 * rq, c0 = sc0 + 4 * cq;
  float4 x[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src + sw_off_h(r0 + a, c0, Rs));
    const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    x[a] = make_float4(lo.x, lo.y, hi.x, hi.y);
  }
  *reinterpret_cast<float4*>(dst + sw_off(roff + c0 + 0, r0, Rd)) = make_float4(x[0].x, x[1].x, x[2].x, x[3].x);
  *reinterpret_cast<float4*>(dst + sw_off(roff + c0 + 1, r0, Rd)) = make_float4(x[0].y, x[1].y, x[2].y, x[3].y);
  *reinterpret_cast<float4*>(dst + sw_off(roff + c0 + 2, r0, Rd)) = make_float4(x[0].z, x[1].z, x[2].z, x[3].z);
  *reinterpret_cast<float4*>(dst + sw_off(roff + c0 + 3, r0, Rd)) = make_float4(x[0].w, x[1].w, x[2].w, x[3].w);
}

__global__ void __launch_bounds__(WALKV_THREADS, 1) k_walk_bwd_v(const __grid_constant__ WalkBwdArgs a) {
  extern __shared__ unsigned char smraw[];
  WalkBvSmem& s = *reinterpret_cast<WalkBvSmem*>(tc::align1024(smraw));
  const int seg = a.seg_base + blockIdx.x / a.HV;  // all heads of the longest document's segments first
  const int h = blockIdx.x % a.HV;
  const SegDesc dd = a.segs[seg];
  const int n = dd.nchunks;
  // What this CTA walks: its segment's full adjoint walk with the outputs
  // (mode 0); in the summary launch (mode 1), by blockIdx.y: 0 the last
  // segment of a split document from dht, giving the end adjoint of the one
  // before; 1 a middle segment from a zero end adjoint (its start adjoint).
  int kind = 0;
  if (a.mode == 1) {
    kind = 1 + (int)blockIdx.y;
    const bool on = blockIdx.y == 0 ? (dd.idx == dd.nseg - 1 && dd.nseg > 1) : (dd.idx >= 1 && dd.idx <= dd.nseg - 2);
    if (!on) return;
  }
  const bool outputs = kind == 0;
  // The chunks of this launch, [mb, me) of the segment walked from me - 1
  // down: all of them, or one slice of a pipelined walk (mb even), which
  // starts from the adjoint the later slice left in the carry buffer and
  // leaves its own there.
  if (kind == 0 && a.m0 > 0 && a.m0 >= n) return;
  const int mb = kind == 0 ? min(a.m0, n) : 0, me = kind == 0 ? min(a.m1, n) : n, cnt = me - mb;
  // Start (end-of-segment) and end (start-of-segment) adjoints: dht / dh0 of the
  // document, or per-segment buffers [NSEG][HV][128][128].
  auto start_adj = [&]() -> const float* {
    const size_t sidx = ((size_t)dd.doc * a.HV + h) * DK * DK, gidx = ((size_t)seg * a.HV + h) * DK * DK;
    if (kind == 0 && me < n) return a.carry + gidx;
    return (kind == 0 && dd.idx < dd.nseg - 1) ? a.dsend + gidx : (kind <= 1 && a.dht ? a.dht + sidx : nullptr);
  };
  auto end_adj = [&]() -> float* {
    const size_t sidx = ((size_t)dd.doc * a.HV + h) * DK * DK, gidx = ((size_t)seg * a.HV + h) * DK * DK;
    if (kind == 0 && mb > 0) return a.carry + gidx;
    return kind == 0   ? (dd.idx == 0 && a.dh0 ? a.dh0 + sidx : nullptr)
           : kind == 1 ? a.dsend + gidx - (size_t)a.HV * DK * DK
                       : a.dsbias + gidx;
  };
  const int tid = threadIdx.x, warp = tid >> 5, lane = lane_id();
  const bool data = tid < 256, issuer = tid == 256;
  const int q4 = warp & 3, hf = (warp >> 2) & 1;
  const int v = 32 * q4 + lane;
  unsigned char* const BA = reinterpret_cast<unsigned char*>(s.BA);
  unsigned char* const BK = reinterpret_cast<unsigned char*>(s.BK);
  unsigned char* const BW = reinterpret_cast<unsigned char*>(s.BW);
  const unsigned char* const SK = reinterpret_cast<const unsigned char*>(s.SK);
  const unsigned char* const SA = reinterpret_cast<const unsigned char*>(s.SA);
  const unsigned char* const SQ = reinterpret_cast<const unsigned char*>(s.SQ);
  const unsigned char* const SW = reinterpret_cast<const unsigned char*>(s.SW);

  if (issuer) {
    tc::mbar_init(&s.bar_k, 1);
    tc::mbar_init(&s.bar_a, 1);
    tc::mbar_init(&s.bar_w, 1);
    tc::mbar_init(&s.bar_ab, 1);
    tc::mbar_init(&s.bar_c, 1);
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
  const uint32_t tl = tm + ((uint32_t)(32 * q4) << 16);

  // Issuer: the staging groups of chunk m.
  auto issue_k = [&](int m) {
    const int item = (dd.chunk0 + m) * a.HV + h;
    tc::mbar_arrive_expect_tx(&s.bar_k, WALKB_K_BYTES);
    tc::tma_load_2d(s.SK, &a.kdt_map, 0, item * DK, &s.bar_k);
    tc::bulk_load(s.gam, &a.gam[(size_t)item * DK], DK * 4, &s.bar_k);
  };
  auto issue_a = [&](int m) {
    const int item = (dd.chunk0 + m) * a.HV + h;
    tc::mbar_arrive_expect_tx(&s.bar_a, WALKB_A_BYTES);
    tc::tma_load_2d(s.SA, &a.aqk_map, 0, item * CH, &s.bar_a);
    for (int kb = 0; kb < 2; ++kb) tc::tma_load_2d(s.SQ + kb * CH * 64, &a.qp_map, kb * 64, item * CH, &s.bar_a);
  };
  auto issue_w = [&](int m) {
    const int item = (dd.chunk0 + m) * a.HV + h;
    tc::mbar_arrive_expect_tx(&s.bar_w, WALKB_W_BYTES);
    for (int kb = 0; kb < 2; ++kb) tc::tma_load_2d(s.SW + kb * CH * 64, &a.w_map, kb * 64, item * CH, &s.bar_w);
  };
  // dO of chunk m, rows i = 32 hf .., at value column v, as raw BF16 bits into
  // registers (loaded a step before use; rows beyond the chunk read its first
  // row and are zeroed when stored), and (scale dO)' into tensor memory.
  auto load_do = [&](int m, uint16_t (&d)[32]) {  // raw BF16 bits; not used before the next step
    const int i0 = 32 * hf, len = min(CH, dd.len - CH * m);
    const uint16_t* dp = reinterpret_cast<const uint16_t*>(a.dout) + ((size_t)(dd.tok0 + CH * m) * a.HV + h) * DK + v;
#pragma unroll
    for (int i = 0; i < 32; ++i) d[i] = __ldg(dp + (size_t)(i0 + i < len ? i0 + i : 0) * a.HV * DK);
  };
  auto store_do = [&](int m, int b, const uint16_t (&d)[32]) {
    const int i0 = 32 * hf, len = min(CH, dd.len - CH * m);
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = i0 + i < len ? tf32(a.scale * bfbits2f(d[i])) : 0u;
    tc::tmem_st32(tl + colDO(b) + 32 * hf, r);
  };

  uint16_t don[32];  // dO of the next step's chunk, loaded a step ahead
  if (data) {
    // dS <- the end adjoint (dht, a merged segment end adjoint or 0),
    // transposed: dS^T[v][c] = start[c][v].
    uint32_t r[32];
    const float* start = start_adj();
#pragma unroll
    for (int cb = 0; cb < 64; cb += 32) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int c = 64 * hf + cb + j;
        r[j] = __float_as_uint(start ? start[(size_t)c * DK + v] : 0.f);
      }
      tc::tmem_st32(tl + kBColS + 64 * hf + cb, r);
    }
    if (cnt > 0) {
      load_do(me - 1, don);
      store_do(me - 1, 0, don);
    }
    if (cnt > 1) load_do(me - 2, don);
    tc::tmem_wait_st();
  }
  int k_iss = 0, a_iss = 0, w_iss = 0, k_got = 0, a_got = 0, w_got = 0, ab_iss = 0, c_iss = 0;
  if (issuer && cnt > 0) {
    issue_k(me - 1), ++k_iss;
    issue_a(me - 1), ++a_iss;
    issue_w(me - 1), ++w_iss;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();

  constexpr uint32_t kIdB = tc::idesc_tf32(128, 64), kIdA = tc::idesc_tf32(128, 192), kIdC = tc::idesc_tf32(128, 128);
  bool ok = true;
  int st = 0;
  for (; st < cnt; ++st) {
    const int b = st & 1;
    const int m = me - 1 - st;
    const int chunk = dd.chunk0 + m;
    if (data) {
      if (st > 0) {
        ok = tc::mbar_wait(&s.bar_c, (st - 1) & 1) && ok;  // the adjoint of this chunk's end state
        tc::tc_fence_after();
      }
      ok = tc::mbar_wait(&s.bar_k, st & 1) && ok;  // Kd^T and gamma of this chunk
      // Kd [j][c] from Kd^T [c][j]: 16 groups.
      for (int g = warp; g < 16; g += 8) transpose_group(SK, DK, 16 * (g >> 1), 32 * (g & 1), BK, CH, 0);
      // Columns 64 hf .. 64 hf + 63 of the adjoint in two halves: the dS tape
      // (chunk-major like the state tape), dS' (TF32, the A operand) and
      // diag(gamma) dS in place (only the later products accumulate into dS;
      // gamma is read from its landing buffer, refilled after the barrier).
      __nv_bfloat16* tp = outputs ? a.dstape + state_off(chunk, h, a.HV) : nullptr;
      const float* gm = s.gam + 64 * hf;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int c0 = 64 * hf + 32 * half;
        uint32_t ds[32], r[32];
        tc::tmem_ld32(tl + kBColS + c0, ds);
        tc::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4 && tp; ++q) {
          __nv_bfloat162 p[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            p[e] = __floats2bfloat162_rn(__uint_as_float(ds[8 * q + 2 * e]), __uint_as_float(ds[8 * q + 2 * e + 1]));
          *reinterpret_cast<uint4*>(tp + tape_off(v, c0 + 8 * q)) = *reinterpret_cast<uint4*>(p);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = tf32(__uint_as_float(ds[j]));
        tc::tmem_st32(tl + kBColSp + c0, r);
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(ds[j]) * gm[32 * half + j]);
        tc::tmem_st32(tl + kBColS + c0, r);
      }
      tc::fence_proxy_async();
      tc::tmem_wait_st();
    }
    tc::tc_fence_before();
    if (!named_sync_and(1, WALKV_THREADS, ok)) break;  // Kd in place; dS', diag(gamma) dS in TMEM
    tc::tc_fence_after();
    if (issuer) {
      ++k_got;
      const uint64_t bk = tc::desc_k_sw128(s.BK);
#pragma unroll
      for (int k = 0; k < DK / 8; ++k)
        tc::mma_tf32_ta(tm + kBColD, tm + kBColSp + 8 * k, tc::kstep32(bk, k, CH), kIdB, k > 0);
      if (st + 1 < cnt) issue_k(m - 1), ++k_iss;  // Kd^T and gamma were read before the barrier
    }
    if (data) {
      ok = tc::mbar_wait(&s.bar_a, st & 1) && ok;  // Aqk, Q Gamma of this chunk
      // Aqk^T [j][i] (8 groups) and Qp^T [c][i] (16 groups) into [Aqk^T ; Qp^T].
      for (int g = warp; g < 24; g += 8) {
        if (g < 8) transpose_group(SA, CH, 16 * (g >> 1), 32 * (g & 1), BA, CH + DK, 0);
        else transpose_group(SQ, CH, 16 * ((g - 8) >> 2), 32 * ((g - 8) & 3), BA, CH + DK, CH);
      }
      if (st + 1 < cnt) store_do(m - 1, b ^ 1, don);
      if (st + 2 < cnt) load_do(m - 2, don);
      tc::fence_proxy_async();
      tc::tmem_wait_st();
    }
    tc::tc_fence_before();
    if (!named_sync_and(3, WALKV_THREADS, ok)) break;  // [Aqk^T ; Qp^T] in place
    tc::tc_fence_after();
    if (issuer) {
      ++a_got;
      const uint64_t ba = tc::desc_k_sw128(s.BA);
#pragma unroll
      for (int k = 0; k < CH / 8; ++k)
        tc::mma_tf32_ta(tm + kBColD, tm + colDO(b) + 8 * k, tc::kstep32(ba, k, CH + DK), kIdA, 1);
      tc::mma_commit(&s.bar_ab);
      ++ab_iss;
      if (st + 1 < cnt) issue_a(m - 1), ++a_iss;
    }
    if (data) {
      ok = tc::mbar_wait(&s.bar_w, st & 1) && ok;  // w of this chunk
      for (int g = warp; g < 16; g += 8) transpose_group(SW, CH, 16 * (g >> 2), 32 * (g & 3), BW, DK, 0);
      tc::fence_proxy_async();
      ok = tc::mbar_wait(&s.bar_ab, st & 1) && ok;
      tc::tc_fence_after();
      uint32_t r[32];
      tc::tmem_ld32(tl + kBColD + 32 * hf, r);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = tf32(-__uint_as_float(r[j]));
      tc::tmem_st32(tl + kBColDn + 32 * hf, r);  // -dDelta' (the FP32 dDelta stays for the store below)
      tc::tmem_wait_st();
    }
    tc::tc_fence_before();
    if (!named_sync_and(2, WALKV_THREADS, ok)) break;  // -dDelta' in TMEM, w^T in place
    tc::tc_fence_after();
    if (data && outputs) {  // the FP32 dDelta for the gradient kernels, while the last product runs
      uint32_t r[32];
      tc::tmem_ld32(tl + kBColD + 32 * hf, r);
      tc::tmem_wait_ld();
      float* dp = a.ddelta + tf_off(chunk, h, a.HV) + (size_t)(32 * hf) * LDF + v;
#pragma unroll
      for (int j = 0; j < 32; ++j) dp[(size_t)j * LDF] = __uint_as_float(r[j]);
    }
    if (issuer) {
      ++w_got;
      const uint64_t bw = tc::desc_k_sw128(s.BW);
#pragma unroll
      for (int k = 0; k < CH / 8; ++k)
        tc::mma_tf32_ta(tm + kBColS, tm + kBColDn + 8 * k, tc::kstep32(bw, k, DK), kIdC, 1);
      tc::mma_commit(&s.bar_c);
      ++c_iss;
      if (st + 1 < cnt) issue_w(m - 1), ++w_iss;
    }
  }
  if (st < cnt) {
    // A wait ran out: record it and drain the copies and products in flight.
    if (issuer) {
      atomicExch(a.err, 4);
      if (k_iss > k_got) tc::mbar_wait(&s.bar_k, (k_iss - 1) & 1);
      if (a_iss > a_got) tc::mbar_wait(&s.bar_a, (a_iss - 1) & 1);
      if (w_iss > w_got) tc::mbar_wait(&s.bar_w, (w_iss - 1) & 1);
      if (ab_iss > 0) tc::mbar_wait(&s.bar_ab, (ab_iss - 1) & 1);
      if (c_iss > 0) tc::mbar_wait(&s.bar_c, (c_iss - 1) & 1);
    }
  } else if (data) {
    if (cnt > 0) {
      ok = tc::mbar_wait(&s.bar_c, (cnt - 1) & 1) && ok;
      tc::tc_fence_after();
    }
    float* end = end_adj();
    if (end && ok) {  // end[c][v] = dS^T[v][c]
      uint32_t r[32];
#pragma unroll
      for (int cb = 0; cb < 64; cb += 32) {
        tc::tmem_ld32(tl + kBColS + 64 * hf + cb, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) end[(size_t)(64 * hf + cb + j) * DK + v] = __uint_as_float(r[j]);
      }
    }
    if (!ok) atomicExch(a.err, 4);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tm, 512);
}

cudaError_t launch_walk_bwd_v(const WalkBwdArgs& a, int nsegs, cudaStream_t st) {
  if (nsegs == 0) return cudaSuccess;
  const size_t sm = sizeof(WalkBvSmem) + 1024;
  cudaFuncSetAttribute(k_walk_bwd_v, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  k_walk_bwd_v<<<dim3(nsegs * a.HV, a.mode == 1 ? 2 : 1), WALKV_THREADS, sm, st>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Merges of the segment states of a split document (one CTA per (segment,
// head, 16-column slice of the state); only a document's first segment with
// at least three segments works; 256 threads, thread (c, half) computes
// channel c of 8 columns).  Segment s's walk maps its start state to
//   S_end = M_s S_start + B_s       (M_s: the end state from the identity
//                                    without u; B_s: from a zero state),
// so the adjoints map back as  dS_start = M_s^T dS_end + dB_s.  FP32 on the
// CUDA cores, each sum in a fixed order.
//   forward:  S_start[s+1] = M_s S_start[s] + B_s,   s = 1 .. nseg-2
//             (S_start[1] from the first segment's summary walk)
//   backward: dS_end[s-1] = M_s^T dS_end[s] + dB_s,  s = nseg-2 .. 1
//             (dS_end[nseg-2] from the last segment's summary walk)
// ---------------------------------------------------------------------------
constexpr int MERGE_LDM = DK + 1;
template <bool BWD>
__global__ void __launch_bounds__(256) k_merge(const MergeArgs a) {
  extern __shared__ float msm[];
  float* Ms = msm;                   // M_s [c][c'], padded rows
  float* Ss = msm + DK * MERGE_LDM;  // the state slice [c][16]
  const int seg = a.seg_base + blockIdx.x / (a.HV * 8);
  const int h = (blockIdx.x / 8) % a.HV, vs = (blockIdx.x % 8) * 16;
  const SegDesc sd = a.segs[seg];
  if (sd.idx != 0 || sd.nseg < 3) return;
  const int tid = threadIdx.x, c = tid >> 1, v0 = 8 * (tid & 1);
  auto at = [&](int g) { return ((size_t)g * a.HV + h) * DK * DK; };
  const int s_first = BWD ? sd.nseg - 2 : 1, s_last = BWD ? 1 : sd.nseg - 2;
  const int step = BWD ? -1 : 1;
  // The first input state slice.
  {
    const float* src = a.state + at(sd.first + s_first);
    for (int e = tid; e < DK * 16; e += 256) Ss[e] = src[(size_t)(e >> 4) * DK + vs + (e & 15)];
  }
  for (int s = s_first;; s += step) {
    const float* M = a.smap + at(sd.first + s);
    for (int e = tid; e < DK * DK / 4; e += 256) {
      const float4 x = reinterpret_cast<const float4*>(M)[e];
      const int r = e >> 5, k = (e & 31) * 4;
      Ms[r * MERGE_LDM + k] = x.x;
      Ms[r * MERGE_LDM + k + 1] = x.y;
      Ms[r * MERGE_LDM + k + 2] = x.z;
      Ms[r * MERGE_LDM + k + 3] = x.w;
    }
    __syncthreads();
    const float* bias = a.bias + at(sd.first + s);
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = bias[(size_t)c * DK + vs + v0 + j];
    for (int k = 0; k < DK; ++k) {
      const float m = BWD ? Ms[k * MERGE_LDM + c] : Ms[c * MERGE_LDM + k];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(m, Ss[k * 16 + v0 + j], acc[j]);
    }
    __syncthreads();
    float* dst = a.state + at(sd.first + s + step);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      dst[(size_t)c * DK + vs + v0 + j] = acc[j];
      Ss[c * 16 + v0 + j] = acc[j];
    }
    if (s == s_last) break;
    __syncthreads();
  }
}

cudaError_t launch_merge(const MergeArgs& a, int nsegs, bool backward, cudaStream_t st) {
  if (nsegs == 0) return cudaSuccess;
  const size_t sm = (DK * MERGE_LDM + DK * 16) * sizeof(float);
  if (backward) {
    cudaFuncSetAttribute(k_merge<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_merge<true><<<nsegs * a.HV * 8, 256, sm, st>>>(a);
  } else {
    cudaFuncSetAttribute(k_merge<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_merge<false><<<nsegs * a.HV * 8, 256, sm, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace gdr
