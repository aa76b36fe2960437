// gdr_fwd.cu -- forward kernels: WY prep, inter-chunk state walk, output.
#include "gdr_chunk.cuh"
#include "gdr_kernels.h"
#include "gdr_tc.cuh"

namespace gdr {

// ---------------------------------------------------------------------------
// Prep (one CTA of 8 warps per (chunk, value head)): gate cumsum, gated Gram
// matrices, T = (I + diag(beta) At)^-1, and the chunk tiles the walk and the
// backward need:  w = T beta (K*Gamma),  u = T beta V,  Qp = Q*Gamma,
// Kd = K*exp(gc_last - gc),  gamma = exp(gc_last),  Aqk, At, T.
// The "prep program" of PR #8638 "perf(cake_gdn_kcp): ... graph-replay
// checkpoint recompute hands its tapes to the backward" (opening description).
// ---------------------------------------------------------------------------
template <bool VEC, typename BetaT>
__global__ void __launch_bounds__(256, 2) k_prep(PrepArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ChunkSmemB& s = *reinterpret_cast<ChunkSmemB*>(smem_raw);
  constexpr int LDK = ChunkSmemB::LD;
  const int chunk = a.chunk_base + blockIdx.x, h = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int hq = h / (a.HV / a.Hqk);
  const int tid = threadIdx.x, warp = tid >> 5;
  load_chunk<VEC, BetaT>(s, a.q, a.k, a.g, reinterpret_cast<const BetaT*>(a.beta), cd.tok0, cd.len, hq, h, a.Hqk,
                         a.HV);
  gram<VEC>(s, a.aqk + aqk_off(chunk, h, a.HV));
  invert(s);
  // At and T for the backward: the values its gradient kernel needs, bit for bit.
  if (a.amat) {
    const size_t qo = ts_off(chunk, h, a.HV);
    for (int e = tid; e < CH * CH / 4; e += blockDim.x) {
      const int i = e >> 4, j4 = (e & 15) * 4;
      *reinterpret_cast<float4*>(&a.amat[qo + i * LDS + j4]) = *reinterpret_cast<const float4*>(&s.At[i * LDS + j4]);
      *reinterpret_cast<float4*>(&a.tmat[qo + i * LDS + j4]) = *reinterpret_cast<const float4*>(&s.T[i * LDS + j4]);
    }
  }
  // Qp, Kd, gamma (elementwise; factors exp(gc) and exp(gc_last - gc) are <= 1).
  // Qp and Kd are only ever MMA operands: stored rounded to TF32.
  const size_t toff = tile_off(chunk, h, a.HV);
  for (int e = tid; e < CH * DK / 4; e += blockDim.x) {  // four channels per thread, one 16-byte store
    const int i = e >> 5, d = (e & 31) * 4;
    float r[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float gl = VEC ? s.G[i * LDT + d + q] : s.gs[i];
      r[q] = __uint_as_float(tf32(s.q(i, d + q) * ex2(gl)));
      if (i == 0) a.gam[((size_t)chunk * a.HV + h) * DK + d + q] = ex2(VEC ? s.G[(CH - 1) * LDT + d + q] : s.gs[CH - 1]);
    }
    *reinterpret_cast<float4*>(&a.qp[qp_off(chunk, h, a.HV) + i * LDF + d]) = make_float4(r[0], r[1], r[2], r[3]);
  }
  // Kd stored transposed, [c][j] (the K-major A operand of the walk's state update).
  // A warp covers rows i = 8k .. 8k+7 of channels d .. d+3 (lane bits 0-2 -> i,
  // 3-4 -> d): shared reads are conflict-free, each 8-lane group writes 32 bytes.
  for (int e = tid; e < CH * DK; e += blockDim.x) {
    const int l = e & 31, w = e >> 5;
    const int i = (l & 7) + 8 * (w & 7), d = 4 * (w >> 3) + (l >> 3);
    const float gl = VEC ? s.G[i * LDT + d] : s.gs[i];
    const float glast = VEC ? s.G[(CH - 1) * LDT + d] : s.gs[CH - 1];
    a.kd[kd_off(chunk, h, a.HV) + d * LDS + i] = __uint_as_float(tf32(s.k(i, d) * ex2(glast - gl)));
  }
  __syncthreads();
  // Q tile <- v rows (async), G tile <- beta * K * Gamma (B of w).
  for (int e = tid; e < CH * DK / 8; e += blockDim.x) {
    const int i = e >> 4, d8 = (e & 15) * 8;
    if (i < cd.len)
      cp_async16(&s.Q[i * LDK + d8], a.v + ((size_t)(cd.tok0 + i) * a.HV + h) * DK + d8);
    else
      *reinterpret_cast<uint4*>(&s.Q[i * LDK + d8]) = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_async_commit();
  for (int e = tid; e < CH * DK; e += blockDim.x) {
    const int i = e >> 7, d = e & 127;
    const float gl = VEC ? s.G[i * LDT + d] : s.gs[i];
    s.G[i * LDT + d] = s.beta[i] * s.k(i, d) * ex2(gl);
  }
  cp_async_wait<0>();
  __syncthreads();
  // w (warps 0-3) and u (warps 4-7) = T B over rows j <= i.  Warp q of a
  // product takes channel half q % 2 of row blocks {3, 0} (q < 2) or {2, 1},
  // so that the four warps do equal work.  B of u, beta_j V_jc, is formed from
  // the BF16 v tile as it is read.
  {
    const int prod = warp >> 2, q = warp & 3, c0 = 64 * (q & 1);
    const int Ia = (q >> 1) ? 2 : 3, Ib = 3 - Ia;
    float* out = prod ? a.u + tf_off(chunk, h, a.HV) : a.w + w_off(chunk, h, a.HV);
    const int ldo = prod ? LDF : LDT;
    auto bw = [&](int j, int c) { return s.G[j * LDT + c]; };
    auto bu = [&](int j, int c) { return s.beta[j] * s.q(j, c); };
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int I = pass ? Ib : Ia, i0 = 16 * I;
      float acc[8][4];
      zero_acc(acc);
      for (int kk = 0; kk < 2 * I + 2; ++kk) {
        if (prod)
          mma_kstep<8>(acc, kk * 8, 0, 8, [&](int i, int j) { return s.T[(i0 + i) * LDS + j]; },
                       [&](int j, int c) { return bu(j, c0 + c); });
        else
          mma_kstep<8>(acc, kk * 8, 0, 8, [&](int i, int j) { return s.T[(i0 + i) * LDS + j]; },
                       [&](int j, int c) { return bw(j, c0 + c); });
      }
      {  // rows i0 + g (+8), channel pairs c0 + 8 nt + 2 t: 8-byte stores
        const int lane = lane_id(), g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr)
            *reinterpret_cast<float2*>(&out[(i0 + g + 8 * hr) * ldo + c0 + nt * 8 + 2 * t]) = make_float2(
                __uint_as_float(tf32(acc[nt][2 * hr])), __uint_as_float(tf32(acc[nt][2 * hr + 1])));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// State walk with the chunk outputs, on the tensor cores (one CTA per
// (document, value head, N-column value slice); the document's chunks in
// order, documents issued longest first).  The FP32 state slice
// S[c][v0 .. v0+N) lives in tensor memory, one channel c per TMEM lane.
// Per chunk:
//   tape <- S0 (BF16 row per thread);  S0 -> swizzled TF32 operand tile;
//   P = w S0                 (tcgen05.mma M = 64 tokens, N, K = 128)
//   Delta = u - P            (rows of P back from TMEM; Delta -> operand tile)
//   S <- diag(gamma) S0 + Kd^T Delta   (gamma applied in TMEM, then
//                            M = 128 channels, N, K = 64 accumulating)
//   O = Qp S0 + Aqk Delta    (M = 64 tokens, N, K = 128 + 64, reusing the
//                            S0 and Delta operand tiles), written out as
//                            scale * O in BF16 during the next chunk.
// Only P and the state update are on the chain from one chunk to the next:
// each is committed on its own.  Qp S0 queues behind P; Aqk Delta of a chunk
// is issued at the head of the next chunk's first batch (ahead of P, which
// is needed later than it is ready), so the state update is the only
// product between forming Delta and the next chunk.
// w, Qp, Kd^T and Aqk of the next chunk are fetched by TMA as soon as this
// chunk's P and Qp S0 are done (w and Qp single-buffered; Kd^T and Aqk into
// the second of two stages, free because the previous chunk's Aqk Delta was
// issued before P); u and gamma one chunk ahead, refilled once Delta is formed.  Waits are bounded; a timed-out
// wait ends the walk for the whole CTA and sets the device error word.
// The "state walk" and "output program" of PR #8638 (opening description)
// and the walks of PR #7723 (opening description), fused.
// ---------------------------------------------------------------------------
template <int N>
struct WalkTcSmem {
  static constexpr int UB = N < 32 ? 1 : N / 32;  // 32-column TMA boxes of the u slice
  float W[CH * DK];         // A of P: w, rows j, K = c (four 64 x 32 column blocks)
  float Qp[CH * DK];        // A of O: Q Gamma, rows i, K = c (four 64 x 32 column blocks)
  float KdT[2][DK * CH];    // A of the update: Kd^T, rows c, K = j (two 128 x 32 column blocks)
  float Aqk[2][CH * CH];    // A of O: Aqk, rows i, K = j (two 64 x 32 column blocks)
  float Sop[N * DK];        // B of P and O: S0, rows v, K = c
  float Dop[N * CH];        // B of the update and O: Delta, rows v, K = j
  float U[CH * 32 * UB];    // u slice, rows j, 32-column swizzled blocks
  float gam[DK];
  uint64_t bar_u, bar_wq, bar_k[2], bar_p, bar_o1, bar_up, bar_o2;
  uint32_t tmem;
};

// 4 data warps (thread t <-> TMEM lane t <-> channel c = t) and one issuer
// warp (warp 4, lane 0) that issues the TMA copies and the MMAs.
template <int N>
__global__ void __launch_bounds__(160) k_walk_fwd(const __grid_constant__ WalkArgs a) {
  constexpr int VS = DK / N;  // CTAs per (doc, head)
  constexpr int UB = WalkTcSmem<N>::UB;
  constexpr uint32_t TCOLS = 4 * N < 32 ? 32 : 4 * N;  // S, P, O[2]
  constexpr uint32_t U_BYTES = (CH * 32 * UB + DK) * 4;
  constexpr uint32_t WQ_BYTES = 2 * CH * DK * 4;
  constexpr uint32_t K_BYTES = (DK * CH + CH * CH) * 4;
  extern __shared__ unsigned char smraw[];
  WalkTcSmem<N>& s = *reinterpret_cast<WalkTcSmem<N>*>(tc::align1024(smraw));
  const int rank = a.rank_base + blockIdx.x / (a.HV * VS);  // all heads and slices of the longest document first
  const int h = (blockIdx.x / VS) % a.HV;
  const int doc = a.order[rank];
  const DocDesc dd = a.docs[doc];
  const int n = dd.nchunks;
  const int tid = threadIdx.x, warp = tid >> 5, lane = lane_id();
  const bool issuer = tid == 128;
  const int v0 = (blockIdx.x % VS) * N;
  const size_t sidx = ((size_t)doc * a.HV + h) * DK * DK;

  if (issuer) {
    tc::mbar_init(&s.bar_u, 1);
    tc::mbar_init(&s.bar_wq, 1);
    tc::mbar_init(&s.bar_k[0], 1);
    tc::mbar_init(&s.bar_k[1], 1);
    tc::mbar_init(&s.bar_p, 1);
    tc::mbar_init(&s.bar_o1, 1);
    tc::mbar_init(&s.bar_up, 1);
    tc::mbar_init(&s.bar_o2, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&s.tmem, TCOLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s.tmem;
  const uint32_t tS = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's lanes; S in columns [0, N)
  const uint32_t tP = tS + N;                                      // P in columns [N, 2N)
  const uint32_t tO = tS + 2 * N;                                  // O[b] in columns [2N + bN, 3N + bN)

  // Issuer only.  Each stage's copies of chunk m land on its barrier.
  auto issue_u = [&](int m) {  // u slice and gamma
    const int chunk = dd.chunk0 + m;
    const int item = chunk * a.HV + h;
    tc::mbar_arrive_expect_tx(&s.bar_u, U_BYTES);
    for (int ub = 0; ub < UB; ++ub) tc::tma_load_2d(&s.U[ub * CH * 32], &a.u_map, v0 + 32 * ub, item * CH, &s.bar_u);
    tc::bulk_load(s.gam, &a.gam[((size_t)chunk * a.HV + h) * DK], DK * 4, &s.bar_u);
  };
  auto issue_wq = [&](int m) {  // w and Q Gamma
    const int item = (dd.chunk0 + m) * a.HV + h;
    tc::mbar_arrive_expect_tx(&s.bar_wq, WQ_BYTES);
    for (int kb = 0; kb < 4; ++kb) {
      tc::tma_load_2d(&s.W[kb * CH * 32], &a.w_map, kb * 32, item * CH, &s.bar_wq);
      tc::tma_load_2d(&s.Qp[kb * CH * 32], &a.qp_map, kb * 32, item * CH, &s.bar_wq);
    }
  };
  auto issue_k = [&](int m) {  // Kd^T and Aqk into stage m & 1
    const int b = m & 1;
    const int item = (dd.chunk0 + m) * a.HV + h;
    tc::mbar_arrive_expect_tx(&s.bar_k[b], K_BYTES);
    for (int kb = 0; kb < 2; ++kb) {
      tc::tma_load_2d(&s.KdT[b][kb * DK * 32], &a.kdt_map, kb * 32, item * DK, &s.bar_k[b]);
      tc::tma_load_2d(&s.Aqk[b][kb * CH * 32], &a.aqk_map, kb * 32, item * CH, &s.bar_k[b]);
    }
  };
  // scale * O of chunk m (TMEM buffer m & 1) -> out, rows below the chunk's length.
  auto write_out = [&](int m) {  // data warps only
    const int i0 = 64 * m, len = min(CH, dd.len - i0);
    uint32_t orr[N / 2];
#pragma unroll
    for (int cb = 0; cb < N; cb += 16)
      tc::tmem_ld16x256b_x2(tO + (m & 1) * N + cb, *reinterpret_cast<uint32_t(*)[8]>(&orr[cb / 2]));
    tc::tmem_wait_ld();
    const int g = lane >> 2, u2 = (lane & 3) * 2;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = 16 * warp + g + 8 * hr;
      if (i < len) {
        __nv_bfloat16* orow = a.out + ((size_t)(dd.tok0 + i0 + i) * a.HV + h) * DK + v0;
#pragma unroll
        for (int q = 0; q < N / 8; ++q)
          *reinterpret_cast<__nv_bfloat162*>(orow + 8 * q + u2) = __floats2bfloat162_rn(
              a.scale * __uint_as_float(orr[4 * q + 2 * hr]), a.scale * __uint_as_float(orr[4 * q + 2 * hr + 1]));
      }
    }
  };
  auto kstep = [](uint64_t desc, int k, int rows) {  // K = 8 step k of a K-major SW128 operand
    return desc + (uint64_t)((((k >> 2) * rows * 128) + (k & 3) * 32) >> 4);
  };

  if (tid < DK) {  // S <- h0 (or 0)
#pragma unroll
    for (int cb = 0; cb < N; cb += 16) {
      uint32_t r[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        r[q] = __float_as_uint(a.h0 ? a.h0[sidx + (size_t)tid * DK + v0 + cb + q] : 0.f);
      tc::tmem_st16(tS + cb, r);
    }
    tc::tmem_wait_st();
  }
  // Copies and output products issued / waited for (issuer), for the drain after a timeout.
  int iss_u = 0, iss_wq = 0, iss_k = 0, got_wq = 0, got_k = 0, o1_iss = 0, o1_done = 0, o2_iss = 0, o2_done = 0;
  if (issuer && n > 0) {
    issue_wq(0), ++iss_wq;
    issue_k(0), ++iss_k;
    issue_u(0), ++iss_u;
  }
  constexpr uint32_t idP = tc::idesc_tf32(CH, N), idU = tc::idesc_tf32(DK, N);
  unsigned char* sop = reinterpret_cast<unsigned char*>(s.Sop);
  unsigned char* dop = reinterpret_cast<unsigned char*>(s.Dop);
  bool ok = true, kprev = false;  // kprev: the previous chunk's Kd^T / Aqk stage was ready
  // O += Aqk Delta of chunk q (issuer; needs Delta of q in the operand tile).
  auto issue_o2 = [&](int q) {
    const uint64_t aa = tc::desc_k_sw128(s.Aqk[q & 1]), bd = tc::desc_k_sw128(s.Dop);
#pragma unroll
    for (int k = 0; k < CH / 8; ++k)
      tc::mma_tf32(tmem + 2 * N + (q & 1) * N, kstep(aa, k, CH), kstep(bd, k, N), idP, 1);
    tc::mma_commit(&s.bar_o2);
    ++o2_iss;
  };
  int m = 0;
  for (; m < n; ++m) {
    const int b = m & 1;
    const int chunk = dd.chunk0 + m;
    const size_t toff = tile_off(chunk, h, a.HV);
    if (issuer) {
      const bool r = tc::mbar_wait(&s.bar_wq, m & 1);
      ok = r && ok;
      got_wq += r;
    }
    uint32_t sr[N];
    if (tid < DK) {
      // S0 row c = tid; S0 as the B operand of P and O (row v, k = c).
#pragma unroll
      for (int cb = 0; cb < N; cb += 16) tc::tmem_ld16(tS + cb, *reinterpret_cast<uint32_t(*)[16]>(&sr[cb]));
      tc::tmem_wait_ld();
#pragma unroll
      for (int v = 0; v < N; ++v)
        *reinterpret_cast<uint32_t*>(sop + tc::sw128_offset(v, tid, N)) = tf32(__uint_as_float(sr[v]));
      tc::fence_proxy_async();
    }
    tc::tc_fence_before();
    if (!__syncthreads_and(ok)) break;
    tc::tc_fence_after();
    if (issuer) {
      // The previous chunk's O += Aqk Delta, then P = w S0 (committed alone:
      // the chain waits on it), then O = Qp S0.
      if (m > 0 && kprev) issue_o2(m - 1);
      const uint64_t aw = tc::desc_k_sw128(s.W), aq = tc::desc_k_sw128(s.Qp), bs = tc::desc_k_sw128(s.Sop);
#pragma unroll
      for (int k = 0; k < DK / 8; ++k) tc::mma_tf32(tmem + N, kstep(aw, k, CH), kstep(bs, k, N), idP, k > 0);
      tc::mma_commit(&s.bar_p);
#pragma unroll
      for (int k = 0; k < DK / 8; ++k)
        tc::mma_tf32(tmem + 2 * N + b * N, kstep(aq, k, CH), kstep(bs, k, N), idP, k > 0);
      tc::mma_commit(&s.bar_o1);
      ++o1_iss;
    }
    if (tid < DK) {
      // While P runs: the tape row, diag(gamma) S0 back into TMEM (columns P
      // does not touch), and the previous chunk's output.
      if (a.tape) {  // S0[c][v0 .. v0+N) as BF16
        uint4* tp = reinterpret_cast<uint4*>(a.tape + state_off(chunk, h, a.HV) + (size_t)tid * DK + v0);
#pragma unroll
        for (int q = 0; q < N; q += 8) {
          __nv_bfloat162 p0 = __floats2bfloat162_rn(__uint_as_float(sr[q]), __uint_as_float(sr[q + 1]));
          __nv_bfloat162 p1 = __floats2bfloat162_rn(__uint_as_float(sr[q + 2]), __uint_as_float(sr[q + 3]));
          __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(sr[q + 4]), __uint_as_float(sr[q + 5]));
          __nv_bfloat162 p3 = __floats2bfloat162_rn(__uint_as_float(sr[q + 6]), __uint_as_float(sr[q + 7]));
          tp[q / 8] = make_uint4(*reinterpret_cast<uint32_t*>(&p0), *reinterpret_cast<uint32_t*>(&p1),
                                 *reinterpret_cast<uint32_t*>(&p2), *reinterpret_cast<uint32_t*>(&p3));
        }
      }
      ok = tc::mbar_wait(&s.bar_u, m & 1) && ok;  // u and gamma of this chunk
      const float gm = s.gam[tid];
#pragma unroll
      for (int v = 0; v < N; ++v) sr[v] = __float_as_uint(__uint_as_float(sr[v]) * gm);
#pragma unroll
      for (int cb = 0; cb < N; cb += 16) tc::tmem_st16(tS + cb, *reinterpret_cast<uint32_t(*)[16]>(&sr[cb]));
      tc::tmem_wait_st();
      if (m > 0) {
        ok = tc::mbar_wait(&s.bar_o2, (m - 1) & 1) && ok;  // O of the previous chunk is complete
        tc::tc_fence_after();
        write_out(m - 1);
      }
      ok = tc::mbar_wait(&s.bar_p, m & 1) && ok;
      tc::tc_fence_after();
      // Delta = u - P over the 16-row block of this warp, spread over all 32 lanes:
      // rows j0 = 16 warp + g and j0 + 8, columns 8q + 2u (+1).
      uint32_t pr[N / 2];
#pragma unroll
      for (int cb = 0; cb < N; cb += 16) tc::tmem_ld16x256b_x2(tP + cb, *reinterpret_cast<uint32_t(*)[8]>(&pr[cb / 2]));
      tc::tmem_wait_ld();
      const int g = lane >> 2, u2 = (lane & 3) * 2;
      const unsigned char* ub = reinterpret_cast<const unsigned char*>(s.U);
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int j = 16 * warp + g + 8 * hr;
        float* drow = a.delta ? a.delta + toff + (size_t)j * DK + v0 : nullptr;
#pragma unroll
        for (int q = 0; q < N / 8; ++q) {
          const int v = 8 * q + u2;
          const float2 uu = *reinterpret_cast<const float2*>(ub + tc::sw128_offset(j, v, CH));
          const float d0 = uu.x - __uint_as_float(pr[4 * q + 2 * hr]);
          const float d1 = uu.y - __uint_as_float(pr[4 * q + 2 * hr + 1]);
          if (drow) *reinterpret_cast<float2*>(drow + v) = make_float2(d0, d1);
          *reinterpret_cast<uint32_t*>(dop + tc::sw128_offset(v, j, N)) = tf32(d0);
          *reinterpret_cast<uint32_t*>(dop + tc::sw128_offset(v + 1, j, N)) = tf32(d1);
        }
      }
      tc::fence_proxy_async();
    } else if (issuer) {
      // Once P and Qp S0 are done, w and Q Gamma are free, and so is the Kd^T /
      // Aqk stage of the previous chunk (its Aqk Delta was issued before P):
      // fetch the next chunk's w, Q Gamma, Kd^T and Aqk (the latter into the
      // stage this chunk's update does not read).
      const bool r = tc::mbar_wait(&s.bar_o1, m & 1);
      ok = r && ok;
      o1_done += r;
      if (r) {
        if (m > 0) ++o2_done;  // covered by this commit
        if (m + 1 < n) {
          issue_wq(m + 1), ++iss_wq;
          issue_k(m + 1), ++iss_k;
        }
      }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (issuer) {
      // The state update (committed alone), then O += Aqk Delta.
      const bool kready = tc::mbar_wait(&s.bar_k[b], (m >> 1) & 1);
      ok = kready && ok;
      if (kready) {
        ++got_k;
        const uint64_t ak = tc::desc_k_sw128(s.KdT[b]), bd = tc::desc_k_sw128(s.Dop);
#pragma unroll
        for (int k = 0; k < CH / 8; ++k) tc::mma_tf32(tmem, kstep(ak, k, DK), kstep(bd, k, N), idU, 1);
      }
      tc::mma_commit(&s.bar_up);
      kprev = kready;
      if (ok && m + 1 < n) issue_u(m + 1), ++iss_u;  // u and gamma were last read before this barrier
    }
    // The data warps wait for the state update before reading S; the issuer
    // too, before refilling the u stage.
    if (tid < DK || issuer) ok = tc::mbar_wait(&s.bar_up, m & 1) && ok;
    tc::tc_fence_after();
  }
  if (m < n) {
    // A wait ran out: record it and drain the copies and products still in flight.
    if (issuer) {
      atomicExch(a.err, 3);
      for (int q = m > 0 ? m - 1 : 0; q < iss_u; ++q) tc::mbar_wait(&s.bar_u, q & 1);
      for (int q = got_wq; q < iss_wq; ++q) tc::mbar_wait(&s.bar_wq, q & 1);
      for (int q = got_k; q < iss_k; ++q) tc::mbar_wait(&s.bar_k[q & 1], (q >> 1) & 1);
      for (int q = o1_done; q < o1_iss; ++q) tc::mbar_wait(&s.bar_o1, q & 1);
      for (int q = o2_done; q < o2_iss; ++q) tc::mbar_wait(&s.bar_o2, q & 1);
    }
  } else {
    if (issuer && n > 0 && kprev) issue_o2(n - 1);  // the last chunk's O += Aqk Delta
    if (tid < DK) {
      if (n > 0) {
        ok = tc::mbar_wait(&s.bar_o2, (n - 1) & 1) && ok;
        tc::tc_fence_after();
        if (ok) write_out(n - 1);
      }
      if (a.ht) {
#pragma unroll
        for (int cb = 0; cb < N; cb += 16) {
          uint32_t r[16];
          tc::tmem_ld16(tS + cb, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 16; ++q) a.ht[sidx + (size_t)tid * DK + v0 + cb + q] = __uint_as_float(r[q]);
        }
      }
      if (!ok) atomicExch(a.err, 3);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TCOLS);
}

// ---------------------------------------------------------------------------
// State walk with the chunk outputs for narrow value slices (N = 16 columns
// per CTA, used when the chains are few enough for 8 CTAs each): the same
// walk as k_walk_fwd with 32 instead of 48 tensor-core products per chunk.
// The FP32 state slice S[c][v0 .. v0+N) lives in tensor memory, one channel c
// per TMEM lane.  Per chunk:
//   S0 -> swizzled TF32 operand tile (rows v, K = c);
//   [P; O] = [w; Qp] S0      one M = 128 product (K = 128): P lands on TMEM
//                            lanes 0..63 (token j), O on lanes 64..127 (token i);
//   Delta = u - P            (one token row per lane; Delta -> operand tile);
//   S <- diag(gamma) S0 + Kd^T Delta   (gamma applied in TMEM while [P; O]
//                            runs; M = 128 channels, K = 64 accumulating);
//   O += Aqk Delta           (M = 128 with the A operand starting 64 rows
//                            before the Aqk tile, so that Aqk's rows meet O's
//                            lanes; the first 64 rows fall on P's lanes,
//                            which are dead by then and overwritten before
//                            their next use);
//   out <- scale * O in BF16 during the next chunk, one token row per lane.
// [P; O], Delta and the state update form the chunk-to-chunk chain.  Aqk
// Delta is issued right after the update; the next chunk's w, Qp, Kd^T, Aqk
// and gamma are fetched by TMA as soon as [P; O] is done, u once Delta is
// formed.  Waits are bounded; a timed-out wait ends the walk for the whole
// CTA and sets the device error word.
// Slices of 64 columns keep k_walk_fwd: there each lane of this layout owns a
// token row, and Delta's and the output's per-row stores cost more than the
// saved products while the walk is close to HBM-bound.
// ---------------------------------------------------------------------------
template <int N>
struct WalkTcSmemS {
  static constexpr int UB = N < 32 ? 1 : N / 32;  // 32-column TMA boxes of the u slice
  float WQ[4][2 * CH * 32];  // A of [P; O]: column block kb = 64 rows of w, then 64 rows of Q Gamma
  float KdT[2][DK * CH];     // A of the update: Kd^T, rows c, K = j (two 128 x 32 column blocks)
  float Aqk[2][CH * CH];     // A of O += Aqk Delta: rows i, K = j (two 64 x 32 column blocks)
  float Sop[N * DK];         // B of [P; O]: S0, rows v, K = c
  float Dop[N * CH];         // B of the update and of Aqk Delta: Delta, rows v, K = j
  float U[CH * 32 * UB];     // u slice, rows j, 32-column swizzled blocks
  float gam[2][DK];          // gamma, with Kd^T and Aqk
  uint64_t bar_u, bar_wq, bar_k[2], bar_p, bar_up, bar_o2;
  uint32_t tmem;
};

// Warps 0..3 (thread t <-> TMEM lane t <-> channel c = t) build the S0 operand
// tile; then warps 0 and 1 form Delta (TMEM lanes 0..63, one token row per
// lane) and warps 2 and 3 write the previous chunk's output (lanes 64..127).
// Warp 4, lane 0 issues the TMA copies and the MMAs.  Warps 5..8 (channel
// c = 32 (warp % 4) + lane) write the tape row and apply diag(gamma) to S in
// TMEM, off the chain.
constexpr int WALK_THREADS_S = 288;
template <int N>
__global__ void __launch_bounds__(WALK_THREADS_S, 1) k_walk_fwd_s(const __grid_constant__ WalkArgs a) {
  constexpr int VS = DK / N;  // CTAs per (doc, head)
  constexpr int UB = WalkTcSmemS<N>::UB;
  constexpr uint32_t TCOLS = 3 * N <= 64 ? 64 : (3 * N <= 128 ? 128 : 256);  // S, [P; O][2]
  constexpr uint32_t U_BYTES = CH * 32 * UB * 4;
  constexpr uint32_t WQ_BYTES = 2 * CH * DK * 4;
  constexpr uint32_t K_BYTES = (DK * CH + CH * CH + DK) * 4;
  extern __shared__ unsigned char smraw[];
  WalkTcSmemS<N>& s = *reinterpret_cast<WalkTcSmemS<N>*>(tc::align1024(smraw));
  const int rank = a.rank_base + blockIdx.x / (a.HV * VS);  // all heads and slices of the longest document first
  const int h = (blockIdx.x / VS) % a.HV;
  const int doc = a.order[rank];
  const DocDesc dd = a.docs[doc];
  const int n = dd.nchunks;
  const int tid = threadIdx.x, warp = tid >> 5, lane = lane_id();
  const bool issuer = tid == 128;
  const bool data = tid < DK, state = tid >= 160;
  const int ch = 32 * (warp & 3) + lane;  // channel (TMEM lane) of a data or state thread
  const int v0 = (blockIdx.x % VS) * N;
  const size_t sidx = ((size_t)doc * a.HV + h) * DK * DK;

  if (issuer) {
    tc::mbar_init(&s.bar_u, 1);
    tc::mbar_init(&s.bar_wq, 1);
    tc::mbar_init(&s.bar_k[0], 1);
    tc::mbar_init(&s.bar_k[1], 1);
    tc::mbar_init(&s.bar_p, 1);
    tc::mbar_init(&s.bar_up, 1);
    tc::mbar_init(&s.bar_o2, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&s.tmem, TCOLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s.tmem;
  const uint32_t tS = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's lanes; S in columns [0, N)
  const uint32_t tPO = tS + N;                                     // [P; O][b] in columns [N + bN, 2N + bN)

  // Issuer only.  Each stage's copies of chunk m land on its barrier.
  auto issue_u = [&](int m) {  // u slice
    const int item = (dd.chunk0 + m) * a.HV + h;
    tc::mbar_arrive_expect_tx(&s.bar_u, U_BYTES);
    for (int ub = 0; ub < UB; ++ub) tc::tma_load_2d(&s.U[ub * CH * 32], &a.u_map, v0 + 32 * ub, item * CH, &s.bar_u);
  };
  auto issue_wq = [&](int m) {  // w and Q Gamma, interleaved by column block
    const int item = (dd.chunk0 + m) * a.HV + h;
    tc::mbar_arrive_expect_tx(&s.bar_wq, WQ_BYTES);
    for (int kb = 0; kb < 4; ++kb) {
      tc::tma_load_2d(&s.WQ[kb][0], &a.w_map, kb * 32, item * CH, &s.bar_wq);
      tc::tma_load_2d(&s.WQ[kb][CH * 32], &a.qp_map, kb * 32, item * CH, &s.bar_wq);
    }
  };
  auto issue_k = [&](int m) {  // Kd^T, Aqk and gamma into stage m & 1
    const int b = m & 1;
    const int item = (dd.chunk0 + m) * a.HV + h;
    tc::mbar_arrive_expect_tx(&s.bar_k[b], K_BYTES);
    for (int kb = 0; kb < 2; ++kb) {
      tc::tma_load_2d(&s.KdT[b][kb * DK * 32], &a.kdt_map, kb * 32, item * DK, &s.bar_k[b]);
      tc::tma_load_2d(&s.Aqk[b][kb * CH * 32], &a.aqk_map, kb * 32, item * CH, &s.bar_k[b]);
    }
    tc::bulk_load(s.gam[b], &a.gam[(size_t)item * DK], DK * 4, &s.bar_k[b]);
  };
  // scale * O of chunk m (TMEM lanes 64.., buffer m & 1) -> out; warps 2 and 3,
  // one token row per lane.
  auto write_out = [&](int m) {
    const int i = 32 * (warp - 2) + lane, len = min(CH, dd.len - 64 * m);
    __nv_bfloat16* orow = a.out + ((size_t)(dd.tok0 + 64 * m + i) * a.HV + h) * DK + v0;
#pragma unroll
    for (int cb = 0; cb < N; cb += 16) {
      uint32_t r[16];
      tc::tmem_ld16(tPO + (m & 1) * N + cb, r);
      tc::tmem_wait_ld();
      if (i < len) {
        uint32_t w[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const __nv_bfloat162 p2 =
              __floats2bfloat162_rn(a.scale * __uint_as_float(r[2 * q]), a.scale * __uint_as_float(r[2 * q + 1]));
          w[q] = *reinterpret_cast<const uint32_t*>(&p2);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) reinterpret_cast<uint32_t*>(orow + cb)[q] = w[q];
      }
    }
  };
  auto kstep = [](uint64_t desc, int k, int rows) {  // K = 8 step k of a K-major SW128 operand
    return desc + (uint64_t)((((k >> 2) * rows * 128) + (k & 3) * 32) >> 4);
  };
  // A descriptor formed at its use: the steps above stay immediates added to
  // it, instead of loop-invariant values held in registers across the walk.
  auto desc_here = [](const void* p) {
    uint64_t d;
    asm volatile("mov.b64 %0, %1;" : "=l"(d) : "l"(tc::desc_k_sw128(p)));
    return d;
  };

  if (data) {  // S <- h0 (or 0)
#pragma unroll
    for (int cb = 0; cb < N; cb += 16) {
      uint32_t r[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        r[q] = __float_as_uint(a.h0 ? a.h0[sidx + (size_t)tid * DK + v0 + cb + q] : 0.f);
      tc::tmem_st16(tS + cb, r);
    }
    tc::tmem_wait_st();
  }
  // Copies and products issued / waited for (issuer), for the drain after a timeout.
  int iss_u = 0, iss_wq = 0, iss_k = 0, got_wq = 0, got_k = 0, p_iss = 0, p_done = 0, o2_iss = 0, o2_done = 0;
  if (issuer && n > 0) {
    issue_wq(0), ++iss_wq;
    issue_k(0), ++iss_k;
    issue_u(0), ++iss_u;
  }
  constexpr uint32_t idM = tc::idesc_tf32(2 * CH, N), idU = tc::idesc_tf32(DK, N);
  unsigned char* sop = reinterpret_cast<unsigned char*>(s.Sop);
  unsigned char* dop = reinterpret_cast<unsigned char*>(s.Dop);
  bool ok = true;
  int m = 0;
  for (; m < n; ++m) {
    const int b = m & 1;
    const int chunk = dd.chunk0 + m;
    const size_t toff = tile_off(chunk, h, a.HV);
    if (issuer) {
      const bool r = tc::mbar_wait(&s.bar_wq, m & 1);
      ok = r && ok;
      got_wq += r;
    }
    if (data) {  // S0 row c = tid as the B operand of [P; O] (row v, k = c)
#pragma unroll
      for (int cb = 0; cb < N; cb += 16) {
        uint32_t sr[16];
        tc::tmem_ld16(tS + cb, sr);
        tc::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q)
          *reinterpret_cast<uint32_t*>(sop + tc::sw128_offset(cb + q, tid, N)) = tf32(__uint_as_float(sr[q]));
      }
      tc::fence_proxy_async();
    }
    tc::tc_fence_before();
    if (!__syncthreads_and(ok)) break;
    tc::tc_fence_after();
    if (issuer) {
      // [P; O] = [w; Qp] S0, committed alone: the chain waits on it.
      const uint64_t aw = desc_here(&s.WQ[0][0]), bs = desc_here(s.Sop);
#pragma unroll
      for (int k = 0; k < DK / 8; ++k) tc::mma_tf32(tmem + N + b * N, kstep(aw, k, 2 * CH), kstep(bs, k, N), idM, k > 0);
      tc::mma_commit(&s.bar_p);
      ++p_iss;
      // Once it is done, w and Q Gamma are free, and so is the Kd^T / Aqk
      // stage of the previous chunk (its products were issued before this
      // commit): fetch the next chunk's w, Q Gamma, Kd^T, Aqk and gamma.
      const bool r = tc::mbar_wait(&s.bar_p, m & 1);
      ok = r && ok;
      p_done += r;
      if (r) {
        o2_done = o2_iss;  // covered by this commit
        if (m + 1 < n) {
          issue_wq(m + 1), ++iss_wq;
          issue_k(m + 1), ++iss_k;
        }
      }
    } else if (state) {
      // While [P; O] runs: the tape row and diag(gamma) S0 back into TMEM.
      ok = tc::mbar_wait(&s.bar_k[b], (m >> 1) & 1) && ok;  // gamma of this chunk
      const float gm = s.gam[b][ch];
      uint4* tp = a.tape ? reinterpret_cast<uint4*>(a.tape + state_off(chunk, h, a.HV) + (size_t)ch * DK + v0) : nullptr;
#pragma unroll
      for (int cb = 0; cb < N; cb += 16) {
        uint32_t sr[16];
        tc::tmem_ld16(tS + cb, sr);
        tc::tmem_wait_ld();
        if (tp) {  // S0[c][v0 .. v0+N) as BF16
#pragma unroll
          for (int q = 0; q < 16; q += 8) {
            __nv_bfloat162 p0 = __floats2bfloat162_rn(__uint_as_float(sr[q]), __uint_as_float(sr[q + 1]));
            __nv_bfloat162 p1 = __floats2bfloat162_rn(__uint_as_float(sr[q + 2]), __uint_as_float(sr[q + 3]));
            __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(sr[q + 4]), __uint_as_float(sr[q + 5]));
            __nv_bfloat162 p3 = __floats2bfloat162_rn(__uint_as_float(sr[q + 6]), __uint_as_float(sr[q + 7]));
            tp[(cb + q) / 8] = make_uint4(*reinterpret_cast<uint32_t*>(&p0), *reinterpret_cast<uint32_t*>(&p1),
                                          *reinterpret_cast<uint32_t*>(&p2), *reinterpret_cast<uint32_t*>(&p3));
          }
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) sr[q] = __float_as_uint(__uint_as_float(sr[q]) * gm);
        tc::tmem_st16(tS + cb, sr);
      }
      tc::tmem_wait_st();
    } else if (warp < 2) {
      // Delta = u - P on token row j = 32 warp + lane (TMEM lane j): into the B
      // operand tile and, in FP32, to HBM.
      ok = tc::mbar_wait(&s.bar_u, m & 1) && ok;  // u of this chunk
      ok = tc::mbar_wait(&s.bar_p, m & 1) && ok;
      tc::tc_fence_after();
      const int j = 32 * warp + lane;
      const unsigned char* ub = reinterpret_cast<const unsigned char*>(s.U);
      float4* drow = a.delta ? reinterpret_cast<float4*>(a.delta + toff + (size_t)j * DK + v0) : nullptr;
#pragma unroll
      for (int cb = 0; cb < N; cb += 16) {
        uint32_t pr[16];
        tc::tmem_ld16(tPO + b * N + cb, pr);
        tc::tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int v = cb + 4 * q4;
          const float4 uu = *reinterpret_cast<const float4*>(ub + tc::sw128_offset(j, v, CH));
          const float d[4] = {uu.x - __uint_as_float(pr[4 * q4]), uu.y - __uint_as_float(pr[4 * q4 + 1]),
                              uu.z - __uint_as_float(pr[4 * q4 + 2]), uu.w - __uint_as_float(pr[4 * q4 + 3])};
#pragma unroll
          for (int e = 0; e < 4; ++e) *reinterpret_cast<uint32_t*>(dop + tc::sw128_offset(v + e, j, N)) = tf32(d[e]);
          if (drow) drow[v / 4] = make_float4(d[0], d[1], d[2], d[3]);
        }
      }
      tc::fence_proxy_async();
    } else if (data) {  // warps 2 and 3: the previous chunk's output
      if (m > 0) {
        ok = tc::mbar_wait(&s.bar_o2, (m - 1) & 1) && ok;
        tc::tc_fence_after();
        write_out(m - 1);
      }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (issuer) {
      // The state update (committed alone), then O += Aqk Delta.
      const bool kready = tc::mbar_wait(&s.bar_k[b], (m >> 1) & 1);
      ok = kready && ok;
      if (kready) {
        ++got_k;
        const uint64_t ak = desc_here(s.KdT[b]), bd = desc_here(s.Dop);
#pragma unroll
        for (int k = 0; k < CH / 8; ++k) tc::mma_tf32(tmem, kstep(ak, k, DK), kstep(bd, k, N), idU, 1);
      }
      tc::mma_commit(&s.bar_up);
      if (kready) {
        // A starts 64 rows (8 KB) before each 64-row column block of Aqk: rows
        // 64..127 of the product are Aqk Delta on O's lanes.
        const uint64_t aa = desc_here(reinterpret_cast<const unsigned char*>(s.Aqk[b]) - CH * 128);
        const uint64_t bd = desc_here(s.Dop);
#pragma unroll
        for (int k = 0; k < CH / 8; ++k) tc::mma_tf32(tmem + N + b * N, kstep(aa, k, CH), kstep(bd, k, N), idM, 1);
        tc::mma_commit(&s.bar_o2);
        ++o2_iss;
      }
      if (ok && m + 1 < n) issue_u(m + 1), ++iss_u;  // u was last read before this barrier
    }
    // Every role waits for the state update before the next chunk reads S.
    if (data || state || issuer) ok = tc::mbar_wait(&s.bar_up, m & 1) && ok;
    tc::tc_fence_after();
  }
  if (m < n) {
    // A wait ran out: record it and drain the copies and products still in flight.
    if (issuer) {
      atomicExch(a.err, 3);
      for (int q = m > 0 ? m - 1 : 0; q < iss_u; ++q) tc::mbar_wait(&s.bar_u, q & 1);
      for (int q = got_wq; q < iss_wq; ++q) tc::mbar_wait(&s.bar_wq, q & 1);
      for (int q = got_k; q < iss_k; ++q) tc::mbar_wait(&s.bar_k[q & 1], (q >> 1) & 1);
      for (int q = p_done; q < p_iss; ++q) tc::mbar_wait(&s.bar_p, q & 1);
      for (int q = o2_done; q < o2_iss; ++q) tc::mbar_wait(&s.bar_o2, q & 1);
    }
  } else {
    if (data && warp >= 2 && n > 0) {  // the last chunk's output
      ok = tc::mbar_wait(&s.bar_o2, (n - 1) & 1) && ok;
      tc::tc_fence_after();
      if (ok) write_out(n - 1);
    }
    if (data && a.ht) {
#pragma unroll
      for (int cb = 0; cb < N; cb += 16) {
        uint32_t r[16];
        tc::tmem_ld16(tS + cb, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q) a.ht[sidx + (size_t)tid * DK + v0 + cb + q] = __uint_as_float(r[q]);
      }
    }
    if ((data || state) && !ok) atomicExch(a.err, 3);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TCOLS);
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
cudaError_t launch_prep(const PrepArgs& a, int nchunks, bool vec, bool beta_bf16, cudaStream_t st) {
  if (nchunks == 0) return cudaSuccess;
  const size_t sm = sizeof(ChunkSmemB);
  dim3 grid(nchunks, a.HV);
  if (vec && beta_bf16) {
    cudaFuncSetAttribute(k_prep<true, __nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_prep<true, __nv_bfloat16><<<grid, 256, sm, st>>>(a);
  } else if (vec) {
    cudaFuncSetAttribute(k_prep<true, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_prep<true, float><<<grid, 256, sm, st>>>(a);
  } else if (beta_bf16) {
    cudaFuncSetAttribute(k_prep<false, __nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_prep<false, __nv_bfloat16><<<grid, 256, sm, st>>>(a);
  } else {
    cudaFuncSetAttribute(k_prep<false, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_prep<false, float><<<grid, 256, sm, st>>>(a);
  }
  return cudaGetLastError();
}

template <int N>
static cudaError_t launch_walk_fwd_n(const WalkArgs& a, int ndocs, cudaStream_t st) {
  const size_t sm = sizeof(WalkTcSmem<N>) + 1024;
  cudaFuncSetAttribute(k_walk_fwd<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  dim3 grid(ndocs * a.HV * (DK / N));
  k_walk_fwd<N><<<grid, 160, sm, st>>>(a);
  return cudaGetLastError();
}

template <int N>
static cudaError_t launch_walk_fwd_s(const WalkArgs& a, int ndocs, cudaStream_t st) {
  const size_t sm = sizeof(WalkTcSmemS<N>) + 1024;
  cudaFuncSetAttribute(k_walk_fwd_s<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  dim3 grid(ndocs * a.HV * (DK / N));
  k_walk_fwd_s<N><<<grid, WALK_THREADS_S, sm, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_walk_fwd(const WalkArgs& a, int ndocs, int cols_per_cta, cudaStream_t st) {
  if (ndocs == 0) return cudaSuccess;
  switch (cols_per_cta) {
    case 16: return launch_walk_fwd_s<16>(a, ndocs, st);
    case 32: return launch_walk_fwd_n<32>(a, ndocs, st);
    default: return launch_walk_fwd_n<64>(a, ndocs, st);
  }
}


}  // namespace gdr
