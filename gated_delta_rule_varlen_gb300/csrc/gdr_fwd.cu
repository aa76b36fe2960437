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
  ChunkSmem& s = *reinterpret_cast<ChunkSmem*>(smem_raw);
  const int chunk = blockIdx.x, h = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int hq = h / (a.HV / a.Hqk);
  load_chunk<VEC, BetaT>(s, a.q, a.k, a.g, reinterpret_cast<const BetaT*>(a.beta), cd.tok0, cd.len, hq, h, a.Hqk,
                         a.HV);
  gram<VEC, true>(s, a.aqk + sq_off(chunk, h, a.HV));
  __syncthreads();
  invert(s);
  // Qp, Kd, gamma (elementwise; factors exp(gc) and exp(gc_last - gc) are <= 1).
  const size_t toff = tile_off(chunk, h, a.HV);
  for (int e = threadIdx.x; e < CH * DK; e += blockDim.x) {
    const int i = e >> 7, d = e & 127;
    const float gl = VEC ? s.G[i * LDT + d] : s.gs[i];
    const float glast = VEC ? s.G[(CH - 1) * LDT + d] : s.gs[CH - 1];
    a.qp[toff + e] = s.Q[i * LDT + d] * ex2(gl);
    a.kd[toff + e] = s.K[i * LDT + d] * ex2(glast - gl);
    if (i == 0) a.gam[((size_t)chunk * a.HV + h) * DK + d] = ex2(glast);
  }
  __syncthreads();
  // Q tile <- beta * K * Gamma
  for (int e = threadIdx.x; e < CH * DK; e += blockDim.x) {
    const int i = e >> 7, d = e & 127;
    const float gl = VEC ? s.G[i * LDT + d] : s.gs[i];
    s.Q[i * LDT + d] = s.beta[i] * s.K[i * LDT + d] * ex2(gl);
  }
  __syncthreads();
  const int I = threadIdx.x >> 5, i0 = 16 * I;
  {
    float acc[16][4];
    zero_acc(acc);
    for (int kk = 0; kk < 2 * I + 2; ++kk)
      mma_kstep<16>(acc, kk * 8, 0, 16, [&](int i, int j) { return s.T[(i0 + i) * LDS + j]; },
                    [&](int j, int c) { return s.Q[j * LDT + c]; });
    acc_foreach(acc, [&](int r, int c, float& x) { a.w[toff + (i0 + r) * DK + c] = x; });
  }
  __syncthreads();
  // K tile <- beta * V
  for (int e = threadIdx.x; e < CH * DK; e += blockDim.x) {
    const int i = e >> 7, d = e & 127;
    s.K[i * LDT + d] = i < cd.len ? s.beta[i] * bf2f(a.v[((size_t)(cd.tok0 + i) * a.HV + h) * DK + d]) : 0.f;
  }
  __syncthreads();
  {
    float acc[16][4];
    zero_acc(acc);
    for (int kk = 0; kk < 2 * I + 2; ++kk)
      mma_kstep<16>(acc, kk * 8, 0, 16, [&](int i, int j) { return s.T[(i0 + i) * LDS + j]; },
                    [&](int j, int c) { return s.K[j * LDT + c]; });
    acc_foreach(acc, [&](int r, int c, float& x) { a.u[toff + (i0 + r) * DK + c] = x; });
  }
}

// ---------------------------------------------------------------------------
// State walk (one CTA per (document, value head, value-column slice), the
// document's chunks in order; documents issued longest first).  Each warp owns
// 16 value columns of the FP32 state, held transposed (S^T: 16 x 128) in
// mma accumulators, and per chunk:
//   tape <- S0;  Delta = u - w S0;  S <- diag(gamma) S0 + Kd^T Delta.
// The "state walk" of PR #8638 (opening description) and the walks of
// PR #7723 (opening description).
// ---------------------------------------------------------------------------
template <int NW>
__global__ void __launch_bounds__(NW * 32) k_walk_fwd(WalkArgs a) {
  constexpr int VS = 8 / NW;         // CTAs per (doc, head)
  constexpr int LDU = NW * 16 + 4;   // row stride of the u slice
  extern __shared__ __align__(16) float smf[];
  float* sW = smf;
  float* sKd = sW + CH * LDT;
  float* sU = sKd + CH * LDT;
  float* sGam = sU + CH * LDU;
  const int doc = a.order[blockIdx.x / VS];
  const int h = blockIdx.y;
  const DocDesc dd = a.docs[doc];
  const int warp = threadIdx.x >> 5;
  const int lane = lane_id(), g = lane >> 2, t = lane & 3;
  const int vcta = (blockIdx.x % VS) * NW * 16;
  const int v0 = vcta + warp * 16;
  const size_t sidx = ((size_t)doc * a.HV + h) * DK * DK;

  float S[16][4];  // S^T rows v0+g(+8), cols c
  acc_foreach(S, [&](int r, int c, float& x) { x = a.h0 ? a.h0[sidx + (size_t)c * DK + v0 + r] : 0.f; });

  for (int m = 0; m < dd.nchunks; ++m) {
    const int chunk = dd.chunk0 + m;
    const size_t toff = tile_off(chunk, h, a.HV);
    __syncthreads();
    for (int e = threadIdx.x; e < CH * DK / 4; e += NW * 32) {
      const int i = e >> 5, c4 = (e & 31) * 4;
      *reinterpret_cast<float4*>(&sW[i * LDT + c4]) = *reinterpret_cast<const float4*>(&a.w[toff + i * DK + c4]);
      *reinterpret_cast<float4*>(&sKd[i * LDT + c4]) = *reinterpret_cast<const float4*>(&a.kd[toff + i * DK + c4]);
    }
    for (int e = threadIdx.x; e < CH * NW * 4; e += NW * 32) {
      const int i = e / (NW * 4), c4 = (e % (NW * 4)) * 4;
      *reinterpret_cast<float4*>(&sU[i * LDU + c4]) =
          *reinterpret_cast<const float4*>(&a.u[toff + i * DK + vcta + c4]);
    }
    for (int e = threadIdx.x; e < DK; e += NW * 32) sGam[e] = a.gam[((size_t)chunk * a.HV + h) * DK + e];
    __syncthreads();
    if (a.tape) {
      float* tp = a.tape + state_off(chunk, h, a.HV);
      acc_foreach(S, [&](int r, int c, float& x) { tp[(size_t)c * DK + v0 + r] = x; });
    }
    // P = S^T w^T   (16 x 64)
    float P[8][4];
    zero_acc(P);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      uint32_t av[4] = {tf32(S[kk][0]), tf32(S[kk][2]), tf32(S[kk][1]), tf32(S[kk][3])};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float2 wv = *reinterpret_cast<const float2*>(&sW[(nt * 8 + g) * LDT + kk * 8 + 2 * t]);
        uint32_t b[2] = {tf32(wv.x), tf32(wv.y)};
        mma8(P[nt], av, b);
      }
    }
    // Delta^T = u^T - P
    acc_foreach(P, [&](int r, int j, float& x) { x = sU[j * LDU + warp * 16 + r] - x; });
    if (a.delta) acc_foreach(P, [&](int r, int j, float& x) { a.delta[toff + (size_t)j * DK + v0 + r] = x; });
    // S^T <- S^T diag(gamma) + Delta^T Kd
    acc_foreach(S, [&](int r, int c, float& x) { x *= sGam[c]; });
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t av[4] = {tf32(P[kk][0]), tf32(P[kk][2]), tf32(P[kk][1]), tf32(P[kk][3])};
      const int j0 = kk * 8 + 2 * t;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        uint32_t b[2] = {tf32(sKd[j0 * LDT + nt * 8 + g]), tf32(sKd[(j0 + 1) * LDT + nt * 8 + g])};
        mma8(S[nt], av, b);
      }
    }
  }
  if (a.ht) acc_foreach(S, [&](int r, int c, float& x) { a.ht[sidx + (size_t)c * DK + v0 + r] = x; });
}

// ---------------------------------------------------------------------------
// Output (one CTA per (chunk, value head)):  O = scale (Qp S0 + Aqk Delta).
// The "output program" of PR #8218 (kcp_fwd_o) and PR #8638.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) k_out(OutArgs a) {
  const int chunk = blockIdx.x, h = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int I = threadIdx.x >> 5, i0 = 16 * I;
  const float* qp = a.qp + tile_off(chunk, h, a.HV);
  const float* S0 = a.tape + state_off(chunk, h, a.HV);
  const float* aqk = a.aqk + sq_off(chunk, h, a.HV);
  const float* dl = a.delta + tile_off(chunk, h, a.HV);
  float acc[16][4];
  zero_acc(acc);
  for (int kk = 0; kk < 16; ++kk)
    mma_kstep<16>(acc, kk * 8, 0, 16, [&](int i, int c) { return __ldg(&qp[(i0 + i) * DK + c]); },
                  [&](int c, int v) { return __ldg(&S0[c * DK + v]); });
  for (int kk = 0; kk < 2 * I + 2; ++kk)
    mma_kstep<16>(acc, kk * 8, 0, 16, [&](int i, int j) { return __ldg(&aqk[(i0 + i) * CH + j]); },
                  [&](int j, int v) { return __ldg(&dl[j * DK + v]); });
  acc_foreach(acc, [&](int r, int c, float& x) {
    const int i = i0 + r;
    if (i < cd.len) a.out[((size_t)(cd.tok0 + i) * a.HV + h) * DK + c] = __float2bfloat16_rn(a.scale * x);
  });
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
cudaError_t launch_prep(const PrepArgs& a, int nchunks, bool vec, bool beta_bf16, cudaStream_t st) {
  if (nchunks == 0) return cudaSuccess;
  const size_t sm = sizeof(ChunkSmem);
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
  constexpr int LDU = NW * 16 + 4;
  const size_t sm = (size_t)(2 * CH * LDT + CH * LDU + DK) * sizeof(float);
  cudaFuncSetAttribute(k_walk_fwd<NW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  dim3 grid(ndocs * (8 / NW), a.HV);
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
  k_out<<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdr
