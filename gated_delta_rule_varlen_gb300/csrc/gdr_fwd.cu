// gdr_fwd.cu -- forward kernels: WY prep, inter-chunk state walk, output.
#include "gdr_chunk.cuh"
#include "gdr_kernels.h"

namespace gdr {

// ---------------------------------------------------------------------------
// Prep (one CTA per (chunk, value head)): gate cumsum, gated Gram matrices,
// T = (I + diag(beta) At)^-1, and the chunk tiles the walk and the output
// need:  w = T beta (K*Gamma),  u = T beta V,  Qp = Q*Gamma,
// Kd = K*exp(gc_last - gc),  gamma = exp(gc_last),  Aqk.
// The "prep program" of PR #8638 "perf(cake_gdn_kcp): ... graph-replay
// checkpoint recompute hands its tapes to the backward" (opening description).
// ---------------------------------------------------------------------------
template <bool VEC, typename BetaT>
__global__ void __launch_bounds__(128) k_prep(PrepArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ChunkSmemB& s = *reinterpret_cast<ChunkSmemB*>(smem_raw);
  constexpr int LDK = ChunkSmemB::LD;
  const int chunk = blockIdx.x, h = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int hq = h / (a.HV / a.Hqk);
  load_chunk<VEC, BetaT>(s, a.q, a.k, a.g, reinterpret_cast<const BetaT*>(a.beta), cd.tok0, cd.len, hq, h, a.Hqk,
                         a.HV);
  gram<VEC, true>(s, a.aqk + sq_off(chunk, h, a.HV));
  __syncthreads();
  invert(s);
  // Qp, Kd, gamma (elementwise; factors exp(gc) and exp(gc_last - gc) are <= 1).
  // Qp and Kd are only ever MMA operands: stored rounded to TF32.
  const size_t toff = tile_off(chunk, h, a.HV);
  for (int e = threadIdx.x; e < CH * DK; e += blockDim.x) {
    const int i = e >> 7, d = e & 127;
    const float gl = VEC ? s.G[i * LDT + d] : s.gs[i];
    const float glast = VEC ? s.G[(CH - 1) * LDT + d] : s.gs[CH - 1];
    a.qp[toff + e] = __uint_as_float(tf32(s.q(i, d) * ex2(gl)));
    a.kd[toff + e] = __uint_as_float(tf32(s.k(i, d) * ex2(glast - gl)));
    if (i == 0) a.gam[((size_t)chunk * a.HV + h) * DK + d] = ex2(glast);
  }
  __syncthreads();
  // Q tile <- v rows (async; used for u), G tile <- beta * K * Gamma (for w).
  for (int e = threadIdx.x; e < CH * DK / 8; e += blockDim.x) {
    const int i = e >> 4, d8 = (e & 15) * 8;
    if (i < cd.len)
      cp_async16(&s.Q[i * LDK + d8], a.v + ((size_t)(cd.tok0 + i) * a.HV + h) * DK + d8);
    else
      *reinterpret_cast<uint4*>(&s.Q[i * LDK + d8]) = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_async_commit();
  for (int e = threadIdx.x; e < CH * DK; e += blockDim.x) {
    const int i = e >> 7, d = e & 127;
    const float gl = VEC ? s.G[i * LDT + d] : s.gs[i];
    s.G[i * LDT + d] = s.beta[i] * s.k(i, d) * ex2(gl);
  }
  __syncthreads();
  const int I = threadIdx.x >> 5, i0 = 16 * I;
  {
    float acc[16][4];
    zero_acc(acc);
    for (int kk = 0; kk < 2 * I + 2; ++kk)
      mma_kstep<16>(acc, kk * 8, 0, 16, [&](int i, int j) { return s.T[(i0 + i) * LDS + j]; },
                    [&](int j, int c) { return s.G[j * LDT + c]; });
    acc_foreach(acc, [&](int r, int c, float& x) { a.w[toff + (i0 + r) * DK + c] = __uint_as_float(tf32(x)); });
  }
  cp_async_wait<0>();
  __syncthreads();
  // G tile <- beta * V
  for (int e = threadIdx.x; e < CH * DK; e += blockDim.x) {
    const int i = e >> 7, d = e & 127;
    s.G[i * LDT + d] = s.beta[i] * s.q(i, d);
  }
  __syncthreads();
  {
    float acc[16][4];
    zero_acc(acc);
    for (int kk = 0; kk < 2 * I + 2; ++kk)
      mma_kstep<16>(acc, kk * 8, 0, 16, [&](int i, int j) { return s.T[(i0 + i) * LDS + j]; },
                    [&](int j, int c) { return s.G[j * LDT + c]; });
    acc_foreach(acc, [&](int r, int c, float& x) { a.u[toff + (i0 + r) * DK + c] = __uint_as_float(tf32(x)); });
  }
}

// ---------------------------------------------------------------------------
// State walk (one CTA per (document, value head, value-column slice), the
// document's chunks in order; documents issued longest first).  Each warp owns
// 16 value columns of the FP32 state, held transposed (S^T: 16 x 128) in
// mma accumulators, and per chunk:
//   tape <- S0 (BF16);  Delta = u - w S0;  S <- diag(gamma) S0 + Kd^T Delta.
// The next chunk's w, Kd, u slice and gamma are copied into the other half of
// a double buffer with cp.async while the current chunk is computed.
// The "state walk" of PR #8638 (opening description) and the walks of
// PR #7723 (opening description).
// ---------------------------------------------------------------------------
template <int NW>
struct WalkFwdStage {
  float W[CH * LDT];
  float Kd[CH * LDT];
  float U[CH * (NW * 16 + 4)];
  float gam[DK];
};

template <int NW>
__global__ void __launch_bounds__(NW * 32) k_walk_fwd(WalkArgs a) {
  constexpr int VS = 8 / NW;         // CTAs per (doc, head)
  constexpr int LDU = NW * 16 + 4;   // row stride of the u slice
  constexpr int NTH = NW * 32;
  using Stage = WalkFwdStage<NW>;
  extern __shared__ __align__(16) unsigned char smraw[];
  Stage* stg = reinterpret_cast<Stage*>(smraw);
  // Block index -> (document rank, head, value slice): all heads and slices
  // of the longest document first.
  const int rank = blockIdx.x / (a.HV * VS);
  const int h = (blockIdx.x / VS) % a.HV;
  const int doc = a.order[rank];
  const DocDesc dd = a.docs[doc];
  const int warp = threadIdx.x >> 5;
  const int lane = lane_id(), g = lane >> 2, t = lane & 3;
  const int vcta = (blockIdx.x % VS) * NW * 16;
  const int v0 = vcta + warp * 16;
  const size_t sidx = ((size_t)doc * a.HV + h) * DK * DK;

  auto issue = [&](int m, Stage& s) {
    const int chunk = dd.chunk0 + m;
    const size_t toff = tile_off(chunk, h, a.HV);
    for (int e = threadIdx.x; e < CH * DK / 4; e += NTH) {
      const int i = e >> 5, c4 = (e & 31) * 4;
      cp_async16(&s.W[i * LDT + c4], &a.w[toff + i * DK + c4]);
      cp_async16(&s.Kd[i * LDT + c4], &a.kd[toff + i * DK + c4]);
    }
    for (int e = threadIdx.x; e < CH * NW * 4; e += NTH) {
      const int i = e / (NW * 4), c4 = (e % (NW * 4)) * 4;
      cp_async16(&s.U[i * LDU + c4], &a.u[toff + i * DK + vcta + c4]);
    }
    for (int e = threadIdx.x; e < DK / 4; e += NTH)
      cp_async16(&s.gam[e * 4], &a.gam[((size_t)chunk * a.HV + h) * DK + e * 4]);
  };

  float S[16][4];  // S^T rows v0+g(+8), cols c
  acc_foreach(S, [&](int r, int c, float& x) { x = a.h0 ? a.h0[sidx + (size_t)c * DK + v0 + r] : 0.f; });

  if (dd.nchunks > 0) issue(0, stg[0]);
  cp_async_commit();
  for (int m = 0; m < dd.nchunks; ++m) {
    const int chunk = dd.chunk0 + m;
    const size_t toff = tile_off(chunk, h, a.HV);
    if (m + 1 < dd.nchunks) issue(m + 1, stg[(m + 1) & 1]);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const Stage& sm = stg[m & 1];
    if (a.tape) {  // S0^T, [v][c], as BF16 pairs
      __nv_bfloat16* tp = a.tape + state_off(chunk, h, a.HV);
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const int c = nt * 8 + 2 * t;
        *reinterpret_cast<__nv_bfloat162*>(&tp[(size_t)(v0 + g) * DK + c]) = __floats2bfloat162_rn(S[nt][0], S[nt][1]);
        *reinterpret_cast<__nv_bfloat162*>(&tp[(size_t)(v0 + g + 8) * DK + c]) =
            __floats2bfloat162_rn(S[nt][2], S[nt][3]);
      }
    }
    // P = S^T w^T   (16 x 64)
    float P[8][4];
    zero_acc(P);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      uint32_t av[4] = {tf32(S[kk][0]), tf32(S[kk][2]), tf32(S[kk][1]), tf32(S[kk][3])};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float2 wv = *reinterpret_cast<const float2*>(&sm.W[(nt * 8 + g) * LDT + kk * 8 + 2 * t]);
        uint32_t b[2] = {__float_as_uint(wv.x), __float_as_uint(wv.y)};  // stored TF32-rounded
        mma8(P[nt], av, b);
      }
    }
    // Delta^T = u^T - P
    acc_foreach(P, [&](int r, int j, float& x) { x = sm.U[j * LDU + warp * 16 + r] - x; });
    if (a.delta) acc_foreach(P, [&](int r, int j, float& x) { a.delta[toff + (size_t)j * DK + v0 + r] = x; });
    // S^T <- S^T diag(gamma) + Delta^T Kd
    acc_foreach(S, [&](int r, int c, float& x) { x *= sm.gam[c]; });
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t av[4] = {tf32(P[kk][0]), tf32(P[kk][2]), tf32(P[kk][1]), tf32(P[kk][3])};
      const int j0 = kk * 8 + 2 * t;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        uint32_t b[2] = {__float_as_uint(sm.Kd[j0 * LDT + nt * 8 + g]),
                         __float_as_uint(sm.Kd[(j0 + 1) * LDT + nt * 8 + g])};
        mma8(S[nt], av, b);
      }
    }
    __syncthreads();
  }
  if (a.ht) acc_foreach(S, [&](int r, int c, float& x) { a.ht[sidx + (size_t)c * DK + v0 + r] = x; });
}

// ---------------------------------------------------------------------------
// Output (one CTA of 8 warps per (chunk, value head)):
//   O = scale (Qp S0 + Aqk Delta),  warp w: rows 16 (w % 4), columns 64 (w / 4).
// Operands are staged in shared memory with cp.async in two groups so that
// the Aqk / Delta copy overlaps the Qp S0 product.
// The "output program" of PR #8218 (kcp_fwd_o) and PR #8638.
// ---------------------------------------------------------------------------
constexpr int LDB = DK + 8;  // row stride (elements) of a [128][128] BF16 shared tile
struct OutSmem {
  uint16_t S0[DK * LDB];
  float Qp[CH * LDT];
  float Aqk[CH * LDS];
  float Dl[CH * LDT];
};

__global__ void __launch_bounds__(256) k_out(OutArgs a) {
  extern __shared__ __align__(16) unsigned char smraw[];
  OutSmem& s = *reinterpret_cast<OutSmem*>(smraw);
  const int chunk = blockIdx.x, h = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int warp = threadIdx.x >> 5, I = warp & 3, i0 = 16 * I, n0 = (warp >> 2) * 64;
  const size_t toff = tile_off(chunk, h, a.HV);
  const __nv_bfloat16* S0 = a.tape + state_off(chunk, h, a.HV);
  const float* aqk = a.aqk + sq_off(chunk, h, a.HV);
  for (int e = threadIdx.x; e < DK * DK / 8; e += 256) {  // S0^T rows
    const int v = e >> 4, c8 = (e & 15) * 8;
    cp_async16(&s.S0[v * LDB + c8], &S0[v * DK + c8]);
  }
  for (int e = threadIdx.x; e < CH * DK / 4; e += 256) {
    const int i = e >> 5, c4 = (e & 31) * 4;
    cp_async16(&s.Qp[i * LDT + c4], &a.qp[toff + i * DK + c4]);
  }
  cp_async_commit();
  for (int e = threadIdx.x; e < CH * CH / 4; e += 256) {
    const int i = e >> 4, c4 = (e & 15) * 4;
    cp_async16(&s.Aqk[i * LDS + c4], &aqk[i * CH + c4]);
  }
  for (int e = threadIdx.x; e < CH * DK / 4; e += 256) {
    const int i = e >> 5, c4 = (e & 31) * 4;
    cp_async16(&s.Dl[i * LDT + c4], &a.delta[toff + i * DK + c4]);
  }
  cp_async_commit();
  cp_async_wait<1>();
  __syncthreads();
  float acc[8][4];
  zero_acc(acc);
  for (int kk = 0; kk < 16; ++kk)
    mma_kstep<8>(acc, kk * 8, 0, 8, [&](int i, int c) { return s.Qp[(i0 + i) * LDT + c]; },
                 [&](int c, int v) { return bfbits2f(s.S0[(n0 + v) * LDB + c]); });
  cp_async_wait<0>();
  __syncthreads();
  for (int kk = 0; kk < 2 * I + 2; ++kk)
    mma_kstep<8>(acc, kk * 8, 0, 8, [&](int i, int j) { return s.Aqk[(i0 + i) * LDS + j]; },
                 [&](int j, int v) { return s.Dl[j * LDT + n0 + v]; });
  acc_foreach(acc, [&](int r, int c, float& x) {
    const int i = i0 + r;
    if (i < cd.len) a.out[((size_t)(cd.tok0 + i) * a.HV + h) * DK + n0 + c] = __float2bfloat16_rn(a.scale * x);
  });
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
    k_prep<true, __nv_bfloat16><<<grid, 128, sm, st>>>(a);
  } else if (vec) {
    cudaFuncSetAttribute(k_prep<true, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_prep<true, float><<<grid, 128, sm, st>>>(a);
  } else if (beta_bf16) {
    cudaFuncSetAttribute(k_prep<false, __nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_prep<false, __nv_bfloat16><<<grid, 128, sm, st>>>(a);
  } else {
    cudaFuncSetAttribute(k_prep<false, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_prep<false, float><<<grid, 128, sm, st>>>(a);
  }
  return cudaGetLastError();
}

template <int NW>
static cudaError_t launch_walk_fwd_nw(const WalkArgs& a, int ndocs, cudaStream_t st) {
  const size_t sm = 2 * sizeof(WalkFwdStage<NW>);
  cudaFuncSetAttribute(k_walk_fwd<NW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  dim3 grid(ndocs * a.HV * (8 / NW));
  k_walk_fwd<NW><<<grid, NW * 32, sm, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_walk_fwd(const WalkArgs& a, int ndocs, int warps_per_cta, cudaStream_t st) {
  if (ndocs == 0) return cudaSuccess;
  switch (warps_per_cta) {
    case 1: return launch_walk_fwd_nw<1>(a, ndocs, st);
    case 2: return launch_walk_fwd_nw<2>(a, ndocs, st);
    case 4: return launch_walk_fwd_nw<4>(a, ndocs, st);
    default: return launch_walk_fwd_nw<8>(a, ndocs, st);
  }
}

cudaError_t launch_out(const OutArgs& a, int nchunks, cudaStream_t st) {
  if (nchunks == 0) return cudaSuccess;
  dim3 grid(nchunks, a.HV);
  const size_t sm = sizeof(OutSmem);
  cudaFuncSetAttribute(k_out, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  k_out<<<grid, 256, sm, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdr
