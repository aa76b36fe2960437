// gdr_bwd.cu -- backward kernels: reverse adjoint walk, state-side gradient
// products, chunk-local gradients, grouped-head reduction.
//
// Chunk backward (adjoints dO of the chunk's outputs and dS of its end state;
// derived from the forward identities in gdr_common.cuh):
//   dDelta = scale Aqk^T dO + Kd dS
//   dS0    = diag(gamma) dS + scale Qp^T dO - w^T dDelta
//   dAqk   = scale tril(dO Delta^T)
//   X = T^T (-dDelta S0^T),  Y = T^T dDelta
//   dA     = -strict_tril(X w^T + Y u^T)
//   dQ     = scale (dO S0^T)*Gamma + [dAqk (x) decay] K
//   dKp'   = beta X*Gamma + beta [dA (x) decay] K          (= dKp * Gamma)
//   dKn'   = [dAqk (x) decay]^T Q + [beta dA (x) decay]^T K  (= dKn / Gamma)
//   dV     = beta Y
//   dbeta  = rowsum(X*Kp) + rowsum(Y*V) + rowsum(dA*At)
//   dK     = dKp' + dKn' + (Delta dS^T) * exp(gc_last - gc)
//   dgc    = Q*dQ + K*dKp' - K*dKn' - Kd*dKd, plus at the last row
//            gamma*rowsum(dS*S0) + colsum(Kd*dKd);   dg = reverse cumsum(dgc)
// where [M (x) decay]_ij = M_ij exp(gc_i - gc_j) per channel.
#include "gdr_chunk.cuh"
#include "gdr_kernels.h"

namespace gdr {

// ---------------------------------------------------------------------------
// Reverse adjoint walk (one CTA per (document, value head, value-column
// slice), chunks in reverse).  Each warp owns 16 value columns of dS^T.
// The "adjoint walk" of PR #7723 "perf(cake_gdn): prefetch offset adjoint
// walk, default LPT segment plan" (opening description).
// ---------------------------------------------------------------------------
template <int NW>
__global__ void __launch_bounds__(NW * 32) k_walk_bwd(WalkBwdArgs a) {
  constexpr int VS = 8 / NW;
  constexpr int LDU = NW * 16 + 4;
  extern __shared__ __align__(16) float smf[];
  float* sAqk = smf;                 // [64][LDS]
  float* sKd = sAqk + CH * LDS;      // [64][LDT]
  float* sQp = sKd + CH * LDT;
  float* sW = sQp + CH * LDT;
  float* sDO = sW + CH * LDT;        // [64][LDU]
  float* sGam = sDO + CH * LDU;
  const int doc = a.order[blockIdx.x / VS];
  const int h = blockIdx.y;
  const DocDesc dd = a.docs[doc];
  const int warp = threadIdx.x >> 5;
  const int lane = lane_id(), g = lane >> 2, t = lane & 3;
  const int vcta = (blockIdx.x % VS) * NW * 16;
  const int v0 = vcta + warp * 16, w16 = warp * 16;
  const size_t sidx = ((size_t)doc * a.HV + h) * DK * DK;

  float S[16][4];  // dS^T rows v0+g(+8), cols c
  acc_foreach(S, [&](int r, int c, float& x) { x = a.dht ? a.dht[sidx + (size_t)c * DK + v0 + r] : 0.f; });

  for (int m = dd.nchunks - 1; m >= 0; --m) {
    const int chunk = dd.chunk0 + m;
    const ChunkDesc cd = a.chunks[chunk];
    const size_t toff = tile_off(chunk, h, a.HV);
    const size_t qoff = sq_off(chunk, h, a.HV);
    __syncthreads();
    for (int e = threadIdx.x; e < CH * DK / 4; e += NW * 32) {
      const int i = e >> 5, c4 = (e & 31) * 4;
      *reinterpret_cast<float4*>(&sKd[i * LDT + c4]) = *reinterpret_cast<const float4*>(&a.kd[toff + i * DK + c4]);
      *reinterpret_cast<float4*>(&sQp[i * LDT + c4]) = *reinterpret_cast<const float4*>(&a.qp[toff + i * DK + c4]);
      *reinterpret_cast<float4*>(&sW[i * LDT + c4]) = *reinterpret_cast<const float4*>(&a.w[toff + i * DK + c4]);
    }
    for (int e = threadIdx.x; e < CH * CH / 4; e += NW * 32) {
      const int i = e >> 4, c4 = (e & 15) * 4;
      *reinterpret_cast<float4*>(&sAqk[i * LDS + c4]) = *reinterpret_cast<const float4*>(&a.aqk[qoff + i * CH + c4]);
    }
    for (int e = threadIdx.x; e < CH * NW * 8; e += NW * 32) {
      const int i = e / (NW * 8), c2 = (e % (NW * 8)) * 2;
      float2 v = make_float2(0.f, 0.f);
      if (i < cd.len)
        v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(
            &a.dout[((size_t)(cd.tok0 + i) * a.HV + h) * DK + vcta + c2]));
      *reinterpret_cast<float2*>(&sDO[i * LDU + c2]) = v;
    }
    for (int e = threadIdx.x; e < DK; e += NW * 32) sGam[e] = a.gam[((size_t)chunk * a.HV + h) * DK + e];
    __syncthreads();
    {
      float* tp = a.dstape + state_off(chunk, h, a.HV);
      acc_foreach(S, [&](int r, int c, float& x) { tp[(size_t)c * DK + v0 + r] = x; });
    }
    // E = dDelta^T (16 x 64) = scale dO^T Aqk + dS^T Kd^T
    float E[8][4];
    zero_acc(E);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int ia = kk * 8 + t, ib = ia + 4;
      uint32_t av[4] = {tf32(sDO[ia * LDU + w16 + g]), tf32(sDO[ia * LDU + w16 + g + 8]),
                        tf32(sDO[ib * LDU + w16 + g]), tf32(sDO[ib * LDU + w16 + g + 8])};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        if (nt <= kk) {
          uint32_t b[2] = {tf32(sAqk[ia * LDS + nt * 8 + g]), tf32(sAqk[ib * LDS + nt * 8 + g])};
          mma8(E[nt], av, b);
        }
      }
    }
    acc_foreach(E, [&](int r, int j, float& x) { x *= a.scale; });
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      uint32_t av[4] = {tf32(S[kk][0]), tf32(S[kk][2]), tf32(S[kk][1]), tf32(S[kk][3])};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float2 kv = *reinterpret_cast<const float2*>(&sKd[(nt * 8 + g) * LDT + kk * 8 + 2 * t]);
        uint32_t b[2] = {tf32(kv.x), tf32(kv.y)};
        mma8(E[nt], av, b);
      }
    }
    acc_foreach(E, [&](int r, int j, float& x) { a.ddelta[toff + (size_t)j * DK + v0 + r] = x; });
    // dS^T <- dS^T diag(gamma) + scale dO^T Qp - dDelta^T w
    acc_foreach(S, [&](int r, int c, float& x) { x *= sGam[c]; });
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int ia = kk * 8 + t, ib = ia + 4;
      uint32_t av[4] = {tf32(a.scale * sDO[ia * LDU + w16 + g]), tf32(a.scale * sDO[ia * LDU + w16 + g + 8]),
                        tf32(a.scale * sDO[ib * LDU + w16 + g]), tf32(a.scale * sDO[ib * LDU + w16 + g + 8])};
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        uint32_t b[2] = {tf32(sQp[ia * LDT + nt * 8 + g]), tf32(sQp[ib * LDT + nt * 8 + g])};
        mma8(S[nt], av, b);
      }
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t av[4] = {tf32(-E[kk][0]), tf32(-E[kk][2]), tf32(-E[kk][1]), tf32(-E[kk][3])};
      const int j0 = kk * 8 + 2 * t;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        uint32_t b[2] = {tf32(sW[j0 * LDT + nt * 8 + g]), tf32(sW[(j0 + 1) * LDT + nt * 8 + g])};
        mma8(S[nt], av, b);
      }
    }
  }
  if (a.dh0) acc_foreach(S, [&](int r, int c, float& x) { a.dh0[sidx + (size_t)c * DK + v0 + r] = x; });
}

// ---------------------------------------------------------------------------
// State-side products (one CTA per (chunk, value head)):
//   dqs = scale dO S0^T,  dw = -dDelta S0^T,  dKd = Delta dS^T,
//   dgam[c] = sum_v dS[c][v] S0[c][v].
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) k_grad_state(GradStateArgs a) {
  const int chunk = blockIdx.x, h = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int I = threadIdx.x >> 5, i0 = 16 * I;
  const int lane = lane_id(), g = lane >> 2, t = lane & 3;
  const size_t toff = tile_off(chunk, h, a.HV);
  const float* S0 = a.tape + state_off(chunk, h, a.HV);
  const float* dS = a.dstape + state_off(chunk, h, a.HV);
  const float* dl = a.delta + toff;
  const float* ddl = a.ddelta + toff;
  auto dO = [&](int i, int v) -> float {
    const int row = i0 + i;
    return row < cd.len ? ldg_bf(&a.dout[((size_t)(cd.tok0 + row) * a.HV + h) * DK + v]) : 0.f;
  };
  {
    float dq[16][4], dw[16][4];
    zero_acc(dq);
    zero_acc(dw);
    for (int kk = 0; kk < 16; ++kk) {
      const int va = kk * 8 + t, vb = va + 4;
      uint32_t aO[4] = {tf32(dO(g, va)), tf32(dO(g + 8, va)), tf32(dO(g, vb)), tf32(dO(g + 8, vb))};
      uint32_t aD[4] = {tf32(__ldg(&ddl[(i0 + g) * DK + va])), tf32(__ldg(&ddl[(i0 + g + 8) * DK + va])),
                        tf32(__ldg(&ddl[(i0 + g) * DK + vb])), tf32(__ldg(&ddl[(i0 + g + 8) * DK + vb]))};
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const int c = nt * 8 + g;
        uint32_t b[2] = {tf32(__ldg(&S0[c * DK + va])), tf32(__ldg(&S0[c * DK + vb]))};
        mma8(dq[nt], aO, b);
        mma8(dw[nt], aD, b);
      }
    }
    acc_foreach(dq, [&](int r, int c, float& x) { a.dqs[toff + (i0 + r) * DK + c] = a.scale * x; });
    acc_foreach(dw, [&](int r, int c, float& x) { a.dw[toff + (i0 + r) * DK + c] = -x; });
  }
  {
    float acc[16][4];
    zero_acc(acc);
    for (int kk = 0; kk < 16; ++kk)
      mma_kstep<16>(acc, kk * 8, 0, 16, [&](int i, int v) { return __ldg(&dl[(i0 + i) * DK + v]); },
                    [&](int v, int c) { return __ldg(&dS[c * DK + v]); });
    acc_foreach(acc, [&](int r, int c, float& x) { a.dkd[toff + (i0 + r) * DK + c] = x; });
  }
  for (int c = I * 32; c < I * 32 + 32; ++c) {
    const float4 x = *reinterpret_cast<const float4*>(&S0[c * DK + lane * 4]);
    const float4 y = *reinterpret_cast<const float4*>(&dS[c * DK + lane * 4]);
    float sum = x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) a.dgam[((size_t)chunk * a.HV + h) * DK + c] = sum;
  }
}

// ---------------------------------------------------------------------------
// Chunk-local gradients (one CTA per (chunk, value head)).  Warp I owns rows
// 16I..16I+15 of every per-row result; dk and the gate adjoint accumulate in
// shared memory, dg is the reverse chunk-local cumsum of dgc.  The
// "fused gradient" / "gate epilogue" stages named on PR #8218.
// ---------------------------------------------------------------------------
struct GradSmem {
  ChunkSmem c;
  float dAqk[CH * LDS];
  float dK[CH * LDT];
  float dG[CH * LDT];
  float dbeta[CH];
  float col[4 * DK];
  float rowsum[CH];
};

template <bool VEC, typename BetaT>
__global__ void __launch_bounds__(128) k_grad(GradArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  GradSmem& sg = *reinterpret_cast<GradSmem*>(smem_raw);
  ChunkSmem& s = sg.c;
  const int chunk = blockIdx.x, h = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int hq = h / (a.HV / a.Hqk);
  const int tid = threadIdx.x;
  const int I = tid >> 5, i0 = 16 * I;
  const int lane = lane_id(), g = lane >> 2, t = lane & 3;
  const size_t toff = tile_off(chunk, h, a.HV);
  if (tid < CH) sg.dbeta[tid] = 0.f;
  load_chunk<VEC, BetaT>(s, a.q, a.k, a.g, reinterpret_cast<const BetaT*>(a.beta), cd.tok0, cd.len, hq, h, a.Hqk,
                         a.HV);
  gram<VEC, false>(s, nullptr);
  __syncthreads();
  invert(s);
  auto gl = [&](int i, int c) -> float { return VEC ? s.G[i * LDT + c] : s.gs[i]; };

  // dAqk = scale tril(dO Delta^T)
  {
    const float* dl = a.delta + toff;
    float acc[8][4];
    zero_acc(acc);
    for (int kk = 0; kk < 16; ++kk)
      mma_kstep<8>(
          acc, kk * 8, 0, 2 * I + 2,
          [&](int i, int v) {
            const int row = i0 + i;
            return row < cd.len ? ldg_bf(&a.dout[((size_t)(cd.tok0 + row) * a.HV + h) * DK + v]) : 0.f;
          },
          [&](int v, int j) { return __ldg(&dl[j * DK + v]); });
    acc_foreach(acc, [&](int r, int col, float& x) {
      sg.dAqk[(i0 + r) * LDS + col] = col <= i0 + r ? a.scale * x : 0.f;
    });
  }

  // X = T^T dw, Y = T^T dDelta (rows of this warp; T^T is upper triangular)
  float X[16][4], Y[16][4];
  zero_acc(X);
  zero_acc(Y);
  {
    const float* dw = a.dw + toff;
    const float* dd = a.ddelta + toff;
    for (int kk = 2 * I; kk < 8; ++kk) {
      const int ja = kk * 8 + t, jb = ja + 4;
      uint32_t av[4] = {tf32(s.T[ja * LDS + i0 + g]), tf32(s.T[ja * LDS + i0 + g + 8]),
                        tf32(s.T[jb * LDS + i0 + g]), tf32(s.T[jb * LDS + i0 + g + 8])};
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const int c = nt * 8 + g;
        uint32_t bx[2] = {tf32(__ldg(&dw[ja * DK + c])), tf32(__ldg(&dw[jb * DK + c]))};
        uint32_t by[2] = {tf32(__ldg(&dd[ja * DK + c])), tf32(__ldg(&dd[jb * DK + c]))};
        mma8(X[nt], av, bx);
        mma8(Y[nt], av, by);
      }
    }
  }
  // Row-local: dV, dbeta (X.Kp + Y.V), dKp' from X.
  {
    float db0 = 0.f, db1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = g + 8 * (r >> 1), c = nt * 8 + 2 * t + (r & 1);
        const int i = i0 + row;
        const float e = ex2(gl(i, c));
        const float kv = s.K[i * LDT + c];
        const float vv = i < cd.len ? ldg_bf(&a.v[((size_t)(cd.tok0 + i) * a.HV + h) * DK + c]) : 0.f;
        const float part = X[nt][r] * kv * e + Y[nt][r] * vv;
        if (row < 8) db0 += part; else db1 += part;
        if (i < cd.len) a.dv[((size_t)(cd.tok0 + i) * a.HV + h) * DK + c] = __float2bfloat16_rn(s.beta[i] * Y[nt][r]);
        const float dkp = s.beta[i] * X[nt][r] * e;
        sg.dK[i * LDT + c] = dkp;
        sg.dG[i * LDT + c] = kv * dkp;
      }
    }
    db0 += __shfl_xor_sync(0xffffffffu, db0, 1);
    db0 += __shfl_xor_sync(0xffffffffu, db0, 2);
    db1 += __shfl_xor_sync(0xffffffffu, db1, 1);
    db1 += __shfl_xor_sync(0xffffffffu, db1, 2);
    if (t == 0) {
      sg.dbeta[i0 + g] += db0;
      sg.dbeta[i0 + g + 8] += db1;
    }
  }
  // dA = -strict_tril(X w^T + Y u^T)  -> overwrites s.T once every warp is done with T.
  float dAacc[8][4];
  zero_acc(dAacc);
  {
    const float* w = a.w + toff;
    const float* u = a.u + toff;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      uint32_t ax[4] = {tf32(X[kk][0]), tf32(X[kk][2]), tf32(X[kk][1]), tf32(X[kk][3])};
      uint32_t ay[4] = {tf32(Y[kk][0]), tf32(Y[kk][2]), tf32(Y[kk][1]), tf32(Y[kk][3])};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        if (nt < 2 * I + 2) {
          const int j = nt * 8 + g;
          const float2 wv = __ldg(reinterpret_cast<const float2*>(&w[j * DK + kk * 8 + 2 * t]));
          const float2 uv = __ldg(reinterpret_cast<const float2*>(&u[j * DK + kk * 8 + 2 * t]));
          uint32_t bw[2] = {tf32(wv.x), tf32(wv.y)};
          uint32_t bu[2] = {tf32(uv.x), tf32(uv.y)};
          mma8(dAacc[nt], ax, bw);
          mma8(dAacc[nt], ay, bu);
        }
      }
    }
  }
  __syncthreads();
  float* sDA = s.T;
  acc_foreach(dAacc, [&](int r, int col, float& x) { sDA[(i0 + r) * LDS + col] = col < i0 + r ? -x : 0.f; });
  __syncthreads();
  if (tid < CH) {
    float acc = 0.f;
    for (int j = 0; j < tid; ++j) acc += sDA[tid * LDS + j] * s.At[tid * LDS + j];
    sg.dbeta[tid] += acc;
  }
  // dKp' += beta [dA (x) decay] K
  {
    float Z[16][4];
    zero_acc(Z);
    left_apply<VEC>(s, sDA, s.K, Z);
    acc_foreach(Z, [&](int r, int c, float& x) {
      const int i = i0 + r;
      const float v = s.beta[i] * x;
      sg.dK[i * LDT + c] += v;
      sg.dG[i * LDT + c] += s.K[i * LDT + c] * v;
    });
  }
  // dQ = dqs * Gamma + [dAqk (x) decay] K
  {
    float Z[16][4];
    zero_acc(Z);
    left_apply<VEC>(s, sg.dAqk, s.K, Z);
    acc_foreach(Z, [&](int r, int c, float& x) {
      const int i = i0 + r;
      const float dq = __ldg(&a.dqs[toff + i * DK + c]) * ex2(gl(i, c)) + x;
      sg.dG[i * LDT + c] += s.Q[i * LDT + c] * dq;
      if (a.dq_part) {
        a.dq_part[toff + i * DK + c] = dq;
      } else if (i < cd.len) {
        a.dq[((size_t)(cd.tok0 + i) * a.Hqk + hq) * DK + c] = __float2bfloat16_rn(dq);
      }
    });
  }
  // dKn' = [dAqk (x) decay]^T Q + [beta dA (x) decay]^T K
  {
    float Z[16][4];
    zero_acc(Z);
    right_apply2<VEC>(s, sg.dAqk, s.Q, sDA, s.K, Z);
    acc_foreach(Z, [&](int r, int c, float& x) {
      const int i = i0 + r;
      sg.dK[i * LDT + c] += x;
      sg.dG[i * LDT + c] -= s.K[i * LDT + c] * x;
    });
  }
  // dKd terms (own rows), column sums of Kd*dKd, then dk.
  {
    const float* dkd = a.dkd + toff;
    const float* kd = a.kd + toff;
    float csum[4] = {0.f, 0.f, 0.f, 0.f};
    for (int rr = 0; rr < 16; ++rr) {
      const int i = i0 + rr;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int c = lane * 4 + q4;
        const float x = __ldg(&dkd[i * DK + c]);
        const float kdv = __ldg(&kd[i * DK + c]);
        const float glast = VEC ? s.G[(CH - 1) * LDT + c] : s.gs[CH - 1];
        sg.dK[i * LDT + c] += x * ex2(glast - gl(i, c));
        sg.dG[i * LDT + c] -= kdv * x;
        csum[q4] += kdv * x;
      }
    }
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) sg.col[I * DK + lane * 4 + q4] = csum[q4];
    __syncwarp();
    for (int rr = 0; rr < 16; ++rr) {
      const int i = i0 + rr;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int c = lane * 4 + q4;
        const float x = sg.dK[i * LDT + c];
        if (a.dk_part) {
          a.dk_part[toff + i * DK + c] = x;
        } else if (i < cd.len) {
          a.dk[((size_t)(cd.tok0 + i) * a.Hqk + hq) * DK + c] = __float2bfloat16_rn(x);
        }
      }
    }
  }
  __syncthreads();
  const float* gam = a.gam + ((size_t)chunk * a.HV + h) * DK;
  const float* dgam = a.dgam + ((size_t)chunk * a.HV + h) * DK;
  if (VEC) {
    if (tid < DK) {
      const int c = tid;
      const float extra = gam[c] * dgam[c] + sg.col[c] + sg.col[DK + c] + sg.col[2 * DK + c] + sg.col[3 * DK + c];
      float acc = extra;
      for (int i = CH - 1; i >= 0; --i) {
        acc += sg.dG[i * LDT + c];
        if (i < cd.len) a.dg[((size_t)(cd.tok0 + i) * a.HV + h) * DK + c] = acc;
      }
    }
  } else {
    if (tid < CH) {
      float acc = 0.f;
      for (int c = 0; c < DK; ++c) acc += sg.dG[tid * LDT + c];
      sg.rowsum[tid] = acc;
    }
    __syncthreads();
    if (tid == 0) {
      float extra = 0.f;
      for (int c = 0; c < DK; ++c)
        extra += gam[c] * dgam[c] + sg.col[c] + sg.col[DK + c] + sg.col[2 * DK + c] + sg.col[3 * DK + c];
      float acc = extra;
      for (int i = CH - 1; i >= 0; --i) {
        acc += sg.rowsum[i];
        if (i < cd.len) a.dg[(size_t)(cd.tok0 + i) * a.HV + h] = acc;
      }
    }
  }
  if (tid < cd.len)
    reinterpret_cast<BetaT*>(a.dbeta)[(size_t)(cd.tok0 + tid) * a.HV + h] = from_f<BetaT>(sg.dbeta[tid]);
}

// dq / dk of a Q/K head = FP32 sum over its value heads, rounded once.
__global__ void __launch_bounds__(256) k_group_reduce(GroupReduceArgs a) {
  const int chunk = blockIdx.x, hq = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int G = a.HV / a.Hqk;
  for (int e = threadIdx.x; e < cd.len * DK; e += blockDim.x) {
    const int i = e >> 7, c = e & 127;
    float sq = 0.f, sk = 0.f;
    for (int gi = 0; gi < G; ++gi) {
      const size_t off = tile_off(chunk, hq * G + gi, a.HV) + (size_t)i * DK + c;
      sq += a.dq_part[off];
      sk += a.dk_part[off];
    }
    const size_t o = ((size_t)(cd.tok0 + i) * a.Hqk + hq) * DK + c;
    a.dq[o] = __float2bfloat16_rn(sq);
    a.dk[o] = __float2bfloat16_rn(sk);
  }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
template <int NW>
static cudaError_t launch_walk_bwd_nw(const WalkBwdArgs& a, int ndocs, cudaStream_t st) {
  constexpr int LDU = NW * 16 + 4;
  const size_t sm = (size_t)(CH * LDS + 3 * CH * LDT + CH * LDU + DK) * sizeof(float);
  cudaFuncSetAttribute(k_walk_bwd<NW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  dim3 grid(ndocs * (8 / NW), a.HV);
  k_walk_bwd<NW><<<grid, NW * 32, sm, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_walk_bwd(const WalkBwdArgs& a, int ndocs, int warps_per_cta, cudaStream_t st) {
  if (ndocs == 0) return cudaSuccess;
  switch (warps_per_cta) {
    case 1: return launch_walk_bwd_nw<1>(a, ndocs, st);
    case 2: return launch_walk_bwd_nw<2>(a, ndocs, st);
    case 4: return launch_walk_bwd_nw<4>(a, ndocs, st);
    default: return launch_walk_bwd_nw<8>(a, ndocs, st);
  }
}

cudaError_t launch_grad_state(const GradStateArgs& a, int nchunks, cudaStream_t st) {
  if (nchunks == 0) return cudaSuccess;
  k_grad_state<<<dim3(nchunks, a.HV), 128, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_grad(const GradArgs& a, int nchunks, bool vec, bool beta_bf16, cudaStream_t st) {
  if (nchunks == 0) return cudaSuccess;
  const size_t sm = sizeof(GradSmem);
  dim3 grid(nchunks, a.HV);
  if (vec && beta_bf16) {
    cudaFuncSetAttribute(k_grad<true, __nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_grad<true, __nv_bfloat16><<<grid, 128, sm, st>>>(a);
  } else if (vec) {
    cudaFuncSetAttribute(k_grad<true, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_grad<true, float><<<grid, 128, sm, st>>>(a);
  } else if (beta_bf16) {
    cudaFuncSetAttribute(k_grad<false, __nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_grad<false, __nv_bfloat16><<<grid, 128, sm, st>>>(a);
  } else {
    cudaFuncSetAttribute(k_grad<false, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_grad<false, float><<<grid, 128, sm, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_group_reduce(const GroupReduceArgs& a, int nchunks, cudaStream_t st) {
  if (nchunks == 0) return cudaSuccess;
  k_group_reduce<<<dim3(nchunks, a.Hqk), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdr
