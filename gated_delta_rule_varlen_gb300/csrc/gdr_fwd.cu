// gdr_fwd.cu -- forward kernel: the WY prep (the state walks are in gdr_walk.cu).
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
  const bool scaled = a.rq != nullptr;  // in-kernel L2 normalization
  if (scaled && tid < CH) {
    const size_t row = (size_t)(cd.tok0 + min(tid, max(cd.len - 1, 0))) * a.Hqk + hq;
    s.rq[tid] = a.rq[row];
    s.rk[tid] = a.rk[row];
  }
  load_chunk<VEC, BetaT>(s, a.q, a.k, a.g, reinterpret_cast<const BetaT*>(a.beta), cd.tok0, cd.len, hq, h, a.Hqk,
                         a.HV);
  gram<VEC>(s, a.aqk + aqk_off(chunk, h, a.HV), scaled);
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
      r[q] = __uint_as_float(tf32(s.q(i, d + q) * (scaled ? s.rq[i] : 1.f) * ex2(gl)));
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
    a.kd[kd_off(chunk, h, a.HV) + d * LDS + i] =
        __uint_as_float(tf32(s.k(i, d) * (scaled ? s.rk[i] : 1.f) * ex2(glast - gl)));
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
    s.G[i * LDT + d] = s.beta[i] * (scaled ? s.rk[i] : 1.f) * s.k(i, d) * ex2(gl);
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
// In-kernel q/k L2 normalization, before the prep: one warp per (token, Q/K
// head) row of q or of k (lane: elements 4 lane .. 4 lane + 3); the sum of
// squares by shuffles in a fixed order; the normalized row in BF16 (the
// inputs the rest of the path reads) and its scale r in FP32 (the backward's
// Jacobian).  The "use_qk_l2norm_in_kernel" option of PR #8638
// "perf(cake_gdn_kcp): ... graph-replay checkpoint recompute hands its tapes
// to the backward" (workload description).
// ---------------------------------------------------------------------------
constexpr float kL2NormEps = 1e-6f;
__global__ void __launch_bounds__(256) k_l2norm(L2NormArgs a) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= 2 * a.rows) return;
  const bool isk = row >= a.rows;
  const int64_t r0 = isk ? row - a.rows : row;
  const __nv_bfloat16* x = (isk ? a.k : a.q) + r0 * DK + 4 * lane_id();
  const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x));
  const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + 2));
  float ss = (x01.x * x01.x + x01.y * x01.y) + (x23.x * x23.x + x23.y * x23.y);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
  const float r = rsqrtf(ss + kL2NormEps);
  __nv_bfloat16* n = (isk ? a.kn : a.qn) + r0 * DK + 4 * lane_id();
  *reinterpret_cast<__nv_bfloat162*>(n) = __floats2bfloat162_rn(x01.x * r, x01.y * r);
  *reinterpret_cast<__nv_bfloat162*>(n + 2) = __floats2bfloat162_rn(x23.x * r, x23.y * r);
  if (lane_id() == 0) (isk ? a.rk : a.rq)[r0] = r;
}

cudaError_t launch_l2norm(const L2NormArgs& a, cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  k_l2norm<<<(unsigned)((2 * a.rows + 7) / 8), 256, 0, st>>>(a);
  return cudaGetLastError();
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

}  // namespace gdr
