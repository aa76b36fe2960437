// gdr_chunk.cuh -- chunk-local building blocks shared by the prep and the
// gradient kernels: tile loads with the gate cumsum, the gated Gram matrices,
// the unit-lower-triangular inverse and the gated "apply" products of the
// backward.  One CTA works on one (chunk, value head); its warps own 16-row
// blocks of every 64-row result (each kernel maps its warps onto the blocks).
#pragma once
#include "gdr_common.cuh"

namespace gdr {

// Shared-memory tiles of one chunk.  K and Q are kept either as FP32 (ET =
// float) or as their exact BF16 input bits (ET = uint16_t, half the space; the
// chunk loads below fill this form).
// LG_ is the row stride of the gate tile; the prep and the gradient kernels
// use 136 (= 8 mod 32), which serves without bank conflicts float2 reads of
// adjacent channels with the row on the group index (the Gram's fragments,
// accumulator positions) and scalar reads with the row on the
// thread-in-group index (B operands of the applies and of w).
template <typename ET, int LG_ = LDT>
struct ChunkSmemT {
  static constexpr int LD = sizeof(ET) == 4 ? LDT : DK + 8;  // row stride (elements) of K and Q
  static constexpr int LG = LG_;
  ET K[CH * LD];      // k (rows >= len are zero)
  ET Q[CH * LD];      // q
  float G[CH * LG];   // per-channel gate: chunk-local cumsum of g, times log2(e)
  float gs[CH];       // scalar gate: chunk-local cumsum of g, times log2(e)
  float beta[CH];
  float At[CH * LDS];  // strict_tril of the gated Gram K K^T (without beta)
  float T[CH * LDS];   // (I + diag(beta) At)^-1
  float tmp[3 * 256];
  float rq[CH], rk[CH];  // in-kernel L2 normalization: row scales of q and k (when used)
  __device__ __forceinline__ float k(int i, int c) const { return elem(K[i * LD + c]); }
  __device__ __forceinline__ float q(int i, int c) const { return elem(Q[i * LD + c]); }
  // Elements (i, c) and (i, c + 1), c even.
  __device__ __forceinline__ float2 k2(int i, int c) const { return pair(&K[i * LD + c]); }
  __device__ __forceinline__ float2 q2(int i, int c) const { return pair(&Q[i * LD + c]); }
  __device__ __forceinline__ float2 g2(int i, int c) const { return *reinterpret_cast<const float2*>(&G[i * LG + c]); }
  static __device__ __forceinline__ float2 pair(const float* p) { return *reinterpret_cast<const float2*>(p); }
  static __device__ __forceinline__ float2 pair(const uint16_t* p) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  static __device__ __forceinline__ float elem(float x) { return x; }
  static __device__ __forceinline__ float elem(uint16_t x) { return bfbits2f(x); }
};
using ChunkSmemB = ChunkSmemT<uint16_t, LDF>;

// Row scalars of one chunk, read into registers by the first half of a chunk
// load (threads tid < CH, row tid) and stored by the second.
struct RowScalars {
  float beta, g;
};

// First half of a chunk load of k, q (of Q/K head hq), the gate and beta of
// value head h for the chunk rows [tok0, tok0+len): the raw BF16 k and q rows
// (and the per-channel gate rows) by 16-byte async copies as one commit group
// (rows >= len are zero-filled), and this thread's row of beta and of the
// scalar gate into registers.  Nothing is waited for, so the caller may work
// on other tiles while the copies land.
template <bool VEC, typename BetaT, int LG>
__device__ RowScalars load_chunk_issue(ChunkSmemT<uint16_t, LG>& s, const __nv_bfloat16* __restrict__ q,
                                       const __nv_bfloat16* __restrict__ k, const float* __restrict__ g,
                                       const BetaT* __restrict__ beta, int tok0, int len, int hq, int h, int Hqk,
                                       int HV) {
  constexpr int LD = ChunkSmemT<uint16_t, LG>::LD;
  const int tid = threadIdx.x;
  for (int e = tid; e < CH * DK / 8; e += blockDim.x) {
    const int i = e >> 4, d8 = (e & 15) * 8;
    if (i < len) {
      const size_t off = ((size_t)(tok0 + i) * Hqk + hq) * DK + d8;
      cp_async16(&s.K[i * LD + d8], k + off);
      cp_async16(&s.Q[i * LD + d8], q + off);
    } else {
      *reinterpret_cast<uint4*>(&s.K[i * LD + d8]) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(&s.Q[i * LD + d8]) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (VEC) {
    for (int e = tid; e < CH * DK / 4; e += blockDim.x) {
      const int i = e >> 5, d4 = (e & 31) * 4;
      if (i < len)
        cp_async16(&s.G[i * LG + d4], g + ((size_t)(tok0 + i) * HV + h) * DK + d4);
      else
        *reinterpret_cast<float4*>(&s.G[i * LG + d4]) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  cp_async_commit();
  RowScalars r{0.f, 0.f};
  if (tid < len && tid < CH) {
    r.beta = to_f<BetaT>(beta[(size_t)(tok0 + tid) * HV + h]);
    if (!VEC) r.g = g[(size_t)(tok0 + tid) * HV + h];
  }
  return r;
}

// Second half: waits for every async copy of this thread, stores the row
// scalars, and forms the chunk-local gate cumsum (base-2 scaled).  Zero gate
// rows past len keep the cumsum flat, so gc at row 63 equals gc at the chunk's
// last token.  Per-channel gate: one thread per channel walks the 64 rows in
// order (measured faster than splitting the rows over more threads, whose
// extra barrier and pass cost more than the shorter chain saves).  Scalar
// gate: one shuffle scan per warp over the 64 rows, then the first warp's
// total added to the second warp's rows (the same order as the tensor-core
// prep of the scalar gate).  Ends with a block barrier.
template <bool VEC, int LG>
__device__ void load_chunk_finish(ChunkSmemT<uint16_t, LG>& s, RowScalars r) {
  const int tid = threadIdx.x;
  cp_async_wait<0>();
  if (tid < CH) {
    s.beta[tid] = r.beta;
    if (!VEC) s.gs[tid] = r.g * LOG2E;
  }
  __syncthreads();
  if (VEC) {
    if (tid < DK) {
      float acc = 0.f;
#pragma unroll 8
      for (int i = 0; i < CH; ++i) {
        acc += s.G[i * LG + tid] * LOG2E;
        s.G[i * LG + tid] = acc;
      }
    }
  } else if (tid < CH) {
    float x = s.gs[tid];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, d);
      if ((tid & 31) >= d) x += y;
    }
    if (tid == 31) s.tmp[0] = x;
    named_sync(1, CH);
    if (tid >= 32) x += s.tmp[0];
    s.gs[tid] = x;
  }
  __syncthreads();
}

// Both halves of a chunk load back to back.
template <bool VEC, typename BetaT, int LG>
__device__ void load_chunk(ChunkSmemT<uint16_t, LG>& s, const __nv_bfloat16* __restrict__ q,
                           const __nv_bfloat16* __restrict__ k, const float* __restrict__ g,
                           const BetaT* __restrict__ beta, int tok0, int len, int hq, int h, int Hqk, int HV) {
  load_chunk_finish<VEC>(s, load_chunk_issue<VEC, BetaT>(s, q, k, g, beta, tok0, len, hq, h, Hqk, HV));
}

// Gated Gram matrices of one chunk,
//   At[i][j]  = sum_c K_ic K_jc exp(gc_ic - gc_jc)   for j <  i (else 0)  -> s.At
//   Aqk[i][j] = sum_c Q_ic K_jc exp(gc_ic - gc_jc)   for j <= i (else 0)  -> aqk (global, [64][64])
// on 8 warps: warp w takes channels [64 hk, +64) (hk = w / 4) and row block
// I = w % 4 (hk = 0) or 3 - w % 4 (hk = 1).  Row block I has 2I + 2 n-tiles and
// warp w issues from the SM sub-partition w % 4, so each sub-partition gets
// 10 n-tiles.
// Per-channel gates use the block factorization described in gdr_common.cuh.
// Each k-step (channels 8 kk .. 8 kk + 7) puts channels 8 kk + 2t and
// 8 kk + 2t + 1 in the k slots t and t + 4 (the order of the terms within a
// step is free), so each fragment pair is one float2 of gates and one BF16
// pair of k or q.
// The upper channel half leaves its partial sums in s.At and s.T (free until
// the inverse); the lower half adds them in, masks, and writes the results.
// Aqk is stored in FP16 (it is only ever an MMA operand), dense rows of 64.
// With `scaled` (in-kernel L2 normalization: the tiles hold the raw q, k and
// s.rq, s.rk their rows' scales) the results are those of the normalized
// rows: At[i][j] rk_i rk_j and Aqk[i][j] rq_i rk_j, in FP32.
template <bool VEC, typename ET, int LG>
__device__ void gram(ChunkSmemT<ET, LG>& s, __half* __restrict__ aqk, bool scaled = false) {
  const int warp = threadIdx.x >> 5, hk = warp >> 2, I = hk ? 3 - (warp & 3) : (warp & 3), i0 = 16 * I;
  const int lane = lane_id(), g = lane >> 2, t = lane & 3;
  const int ra = i0 + g, rb = i0 + g + 8;
  const float* G = s.G;
  // n-tiles [0, 2I + 2) of row block I (the rest is zero).
  float accK[8][4], accQ[8][4];
  zero_acc(accK);
  zero_acc(accQ);
  if (VEC) {
    auto g2 = [&](int i, int c) { return *reinterpret_cast<const float2*>(&G[i * LG + c]); };
#pragma unroll 2
    for (int kk = 8 * hk; kk < 8 * hk + 8; ++kk) {
      const int c = kk * 8 + 2 * t;
      // Reference: gc at row i0 + 7, for the diagonal and the earlier blocks alike.
      const float2 m = g2(i0 + 7, c), ga = g2(ra, c), gb = g2(rb, c);
      const float e00 = ex2(ga.x - m.x), e10 = ex2(gb.x - m.x), e01 = ex2(ga.y - m.y), e11 = ex2(gb.y - m.y);
      const float2 ka = s.k2(ra, c), kb = s.k2(rb, c), qa = s.q2(ra, c), qb = s.q2(rb, c);
      uint32_t aK[4] = {tf32(ka.x * e00), tf32(kb.x * e10), tf32(ka.y * e01), tf32(kb.y * e11)};
      uint32_t aQ[4] = {tf32(qa.x * e00), tf32(qb.x * e10), tf32(qa.y * e01), tf32(qb.y * e11)};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        if (nt < 2 * I + 2) {
          const int j = nt * 8 + g;
          const float2 gj = g2(j, c), kj = s.k2(j, c);
          uint32_t b[2] = {tf32(kj.x * ex2(m.x - gj.x)), tf32(kj.y * ex2(m.y - gj.y))};
          mma8(accK[nt], aK, b);
          mma8(accQ[nt], aQ, b);
        }
      }
    }
  } else {
#pragma unroll 2
    for (int kk = 8 * hk; kk < 8 * hk + 8; ++kk) {
      const int c0 = kk * 8 + t, c1 = c0 + 4;
      uint32_t aK[4] = {tf32(s.k(ra, c0)), tf32(s.k(rb, c0)), tf32(s.k(ra, c1)), tf32(s.k(rb, c1))};
      uint32_t aQ[4] = {tf32(s.q(ra, c0)), tf32(s.q(rb, c0)), tf32(s.q(ra, c1)), tf32(s.q(rb, c1))};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        if (nt < 2 * I + 2) {
          const int j = nt * 8 + g;
          uint32_t b[2] = {tf32(s.k(j, c0)), tf32(s.k(j, c1))};
          mma8(accK[nt], aK, b);
          mma8(accQ[nt], aQ, b);
        }
      }
    }
  }
  float* tq = s.T;  // partial Aqk of the upper channel half
  if (hk == 1) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = i0 + g + 8 * (r >> 1), col = nt * 8 + 2 * t + (r & 1);
        if (nt < 2 * I + 2) {
          s.At[row * LDS + col] = accK[nt][r];
          tq[row * LDS + col] = accQ[nt][r];
        }
      }
  }
  __syncthreads();
  if (hk == 0) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = i0 + g + 8 * (r >> 1), col = nt * 8 + 2 * t + (r & 1);
        float vK = 0.f, vQ = 0.f;
        if (nt < 2 * I + 2 && col <= row) {
          vK = accK[nt][r] + s.At[row * LDS + col];
          vQ = accQ[nt][r] + tq[row * LDS + col];
          if (!VEC) {
            const float dec = ex2(s.gs[row] - s.gs[col]);
            vK *= dec;
            vQ *= dec;
          }
          if (col == row) vK = 0.f;
          if (scaled) {
            vK *= s.rk[row] * s.rk[col];
            vQ *= s.rq[row] * s.rk[col];
          }
        }
        s.At[row * LDS + col] = vK;
        aqk[row * CH + col] = __float2half_rn(vQ);
      }
  }
  __syncthreads();
}

// s.T = (I + diag(beta) At)^-1, unit lower triangular, in FP32 on CUDA cores,
// on 8 warps.  Diagonal 16x16 blocks by forward substitution (warp I < 4,
// one column per lane of its first 16), then the blocks below them column
// block by column block: six warps (J, half), J < 3, take columns
// [16 J + 8 half, +8) of column block J and compute, for I = J+1 .. 3 in order,
//   T_IJ = -T_II * diag(beta_I) * sum_{K=J}^{I-1} At_IK T_KJ,
// which needs only blocks of those columns that the same warp made before,
// so the off-diagonal part synchronizes within the warp only.  Column block J
// makes 3 - J blocks, so the two J = 0 warps go to different SM
// sub-partitions (warp w issues from w % 4): warp w of half w / 4 takes
// J = w (first half) or J = 7 - w (second half) when that is below 3, so
// warps 0 and 7 take J = 0, 1 and 6 J = 1, 2 and 5 J = 2; 3 and 4 wait.
// At, T: [64][LDS] shared tiles; beta: [64]; tmp: 6 x 128 floats of scratch.
__device__ __forceinline__ void invert_tiles(const float* __restrict__ At, float* __restrict__ T,
                                             const float* __restrict__ beta, float* __restrict__ tmp_all) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = lane_id();
  if (warp < 4 && lane < 16) {
    const int i0 = warp * 16, j = lane;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = (i == j) ? 1.f : 0.f;
      const float bi = beta[i0 + i];
#pragma unroll
      for (int m = 0; m < i; ++m) acc -= bi * At[(i0 + i) * LDS + i0 + m] * x[m];
      x[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) T[(i0 + i) * LDS + i0 + j] = x[i];
  }
  // Zero the strictly upper blocks.
  for (int e = tid; e < CH * CH; e += blockDim.x) {
    const int i = e >> 6, j = e & 63;
    if ((j >> 4) > (i >> 4)) T[i * LDS + j] = 0.f;
  }
  __syncthreads();
  const int half = warp >> 2, J = half ? 7 - warp : warp;
  if (J < 3) {
    // Warp (J, half): the 16 x 8 tile of columns n0 .. n0 + 7 of T_IJ as
    // split-TF32 tensor-core products (hi*hi + hi*lo + lo*hi, about FP32
    // accuracy, in three m16n8k8 accumulators): C = At_I,[16J, 16I)
    // T_[16J, 16I),J, then X = diag(beta_I) C through shared memory into the B
    // layout, then T_IJ = -T_II X.
    const int n0 = 16 * J + 8 * half;
    const int g = lane >> 2, t = lane & 3;
    float* xs = tmp_all + (half * 3 + J) * 128;  // X [16][8]
    for (int I = J + 1; I < 4; ++I) {
      const int r0 = 16 * I;
      float c3[3][4] = {};
      for (int k0 = 16 * J; k0 < r0; k0 += 8) {
        const float a[4] = {At[(r0 + g) * LDS + k0 + t], At[(r0 + g + 8) * LDS + k0 + t],
                            At[(r0 + g) * LDS + k0 + t + 4], At[(r0 + g + 8) * LDS + k0 + t + 4]};
        const float b[2] = {T[(k0 + t) * LDS + n0 + g], T[(k0 + t + 4) * LDS + n0 + g]};
        mma8_split3(c3, a, b);
      }
      float c[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) c[e] = (c3[0][e] + c3[1][e]) + c3[2][e];
      xs[g * 8 + 2 * t] = beta[r0 + g] * c[0];
      xs[g * 8 + 2 * t + 1] = beta[r0 + g] * c[1];
      xs[(g + 8) * 8 + 2 * t] = beta[r0 + g + 8] * c[2];
      xs[(g + 8) * 8 + 2 * t + 1] = beta[r0 + g + 8] * c[3];
      __syncwarp();
      float o3[3][4] = {};
#pragma unroll
      for (int k0 = 0; k0 < 16; k0 += 8) {
        const float a[4] = {T[(r0 + g) * LDS + r0 + k0 + t], T[(r0 + g + 8) * LDS + r0 + k0 + t],
                            T[(r0 + g) * LDS + r0 + k0 + t + 4], T[(r0 + g + 8) * LDS + r0 + k0 + t + 4]};
        const float b[2] = {xs[(k0 + t) * 8 + g], xs[(k0 + t + 4) * 8 + g]};
        mma8_split3(o3, a, b);
      }
      float o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = (o3[0][e] + o3[1][e]) + o3[2][e];
      *reinterpret_cast<float2*>(&T[(r0 + g) * LDS + n0 + 2 * t]) = make_float2(-o[0], -o[1]);
      *reinterpret_cast<float2*>(&T[(r0 + g + 8) * LDS + n0 + 2 * t]) = make_float2(-o[2], -o[3]);
      __syncwarp();
    }
  }
  __syncthreads();
}

template <typename ET, int LG>
__device__ void invert(ChunkSmemT<ET, LG>& s) {
  invert_tiles(s.At, s.T, s.beta, s.tmp);
}

// Two left applies that share Y: Z0_i += sum_{j<=i} M0_ij Y_j exp(gc_i - gc_j),
// Z1 likewise with M1, over the rows i of block I (16I .. 16I+15) and channels
// c0 .. c0 + 8 NT - 1; M0, M1 are masked [64][64] shared tiles, fy(j, c)
// returns Y_jc.  Each gated Y fragment is formed once and feeds both products.
// With a scalar gate (VEC false) M0 and M1 already carry exp(gc_i - gc_j).
template <bool VEC, int NT, typename ET, int LG, class FY>
__device__ void left_apply2(const ChunkSmemT<ET, LG>& s, const float* __restrict__ M0, const float* __restrict__ M1, FY fy,
                            float (&Z0)[NT][4], float (&Z1)[NT][4], int I, int c0) {
  const int i0 = 16 * I;
  const int lane = lane_id(), g = lane >> 2, t = lane & 3;
  if (VEC) {
    float acc0[NT][4], acc1[NT][4];
    auto afrag = [&](const float* M, int j0, int j1, uint32_t (&a)[4]) {
      a[0] = tf32(M[(i0 + g) * LDS + j0]);
      a[1] = tf32(M[(i0 + g + 8) * LDS + j0]);
      a[2] = tf32(M[(i0 + g) * LDS + j1]);
      a[3] = tf32(M[(i0 + g + 8) * LDS + j1]);
    };
    zero_acc(acc0);
    zero_acc(acc1);
    float mI[NT];  // reference gc at row 16I + 7 of this thread's B columns
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mI[nt] = s.G[(i0 + 7) * LG + c0 + nt * 8 + g];
#pragma unroll 2
    for (int kk = 0; kk < 2 * I + 2; ++kk) {  // j in [0, 16I + 16)
      const int j0 = kk * 8 + t, j1 = j0 + 4;
      uint32_t a0[4], a1[4];
      afrag(M0, j0, j1, a0);
      afrag(M1, j0, j1, a1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int c = c0 + nt * 8 + g;
        uint32_t b[2] = {tf32(fy(j0, c) * ex2(mI[nt] - s.G[j0 * LG + c])),
                         tf32(fy(j1, c) * ex2(mI[nt] - s.G[j1 * LG + c]))};
        mma8(acc0[nt], a0, b);
        mma8(acc1[nt], a1, b);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = g + 8 * (r >> 1), col = nt * 8 + 2 * t + (r & 1);
        const float e = ex2(s.G[(i0 + row) * LG + c0 + col] - s.G[(i0 + 7) * LG + c0 + col]);
        Z0[nt][r] += acc0[nt][r] * e;
        Z1[nt][r] += acc1[nt][r] * e;
      }
  } else {
    // Scalar gate: M0 and M1 arrive with the decay exp(gc_i - gc_j) applied.
    const int ra = i0 + g, rb = i0 + g + 8;
#pragma unroll 2
    for (int kk = 0; kk < 2 * I + 2; ++kk) {
      const int j0 = kk * 8 + t, j1 = j0 + 4;
      uint32_t a0[4] = {tf32(M0[ra * LDS + j0]), tf32(M0[rb * LDS + j0]), tf32(M0[ra * LDS + j1]),
                        tf32(M0[rb * LDS + j1])};
      uint32_t a1[4] = {tf32(M1[ra * LDS + j0]), tf32(M1[rb * LDS + j0]), tf32(M1[ra * LDS + j1]),
                        tf32(M1[rb * LDS + j1])};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int c = c0 + nt * 8 + g;
        uint32_t b[2] = {tf32(fy(j0, c)), tf32(fy(j1, c))};
        mma8(Z0[nt], a0, b);
        mma8(Z1[nt], a1, b);
      }
    }
  }
}

// Z_j += sum_{i>=j} (M0_ij Q_i + beta_i M1_ij K_i) * exp(gc_i - gc_j) for rows
// j of block J and channels c0 .. c0 + 31 (four n-tiles).  M0, M1 masked
// [64][64] shared tiles; Q, K the chunk's BF16 tiles.  With a scalar gate (VEC
// false) M0 and M1 already carry exp(gc_i - gc_j).
// Each k-step (rows i = 8 kk .. 8 kk + 7) takes the B fragments of all four
// n-tiles of Q, and of K, from one transposing matrix load each, which hands
// thread (g, t) rows 8 kk + 2t and 8 kk + 2t + 1 of channel c0 + 8 nt + g.  So
// the step's k slots t and t + 4 stand for those two rows (the order of the
// terms within a step is free), and the A fragments (M0, M1 read down a column)
// follow the same assignment; with the [64][68] tiles those reads are free of
// bank conflicts.
template <bool VEC, int NT, int LG>
__device__ void right_apply2(const ChunkSmemT<uint16_t, LG>& s, const float* __restrict__ M0,
                             const float* __restrict__ M1, float (&Z)[NT][4], int J, int c0) {
  static_assert(NT == 4, "one x4 matrix load covers four n-tiles");
  constexpr int LD = ChunkSmemT<uint16_t, LG>::LD;
  const int j0b = 16 * J;
  const int lane = lane_id(), g = lane >> 2, t = lane & 3;
  const int ja = j0b + g, jb = ja + 8;
  // This lane's row of the four 8 x 8 matrices (n-tile lane / 8, row lane % 8).
  const uint16_t* const qrow = s.Q + (lane & 7) * LD + c0 + 8 * (lane >> 3);
  const uint16_t* const krow = s.K + (lane & 7) * LD + c0 + 8 * (lane >> 3);
  float acc[NT][4];  // VEC only: the sums before the row factors
  if (VEC) zero_acc(acc);
  auto& dst = VEC ? acc : Z;
  float mJ[NT];  // VEC: reference gc at row 16J + 7, for block J and the later blocks alike
  const int mref = j0b + 7;
  if (VEC) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mJ[nt] = s.G[mref * LG + c0 + nt * 8 + g];
  }
#pragma unroll 2
  for (int kk = 2 * J; kk < 8; ++kk) {  // i in block J and after
    const int ia = kk * 8 + 2 * t, ib = ia + 1;
    uint32_t yq[4], yk[4];
    ldsm_x4_trans(yq, qrow + kk * 8 * LD);
    ldsm_x4_trans(yk, krow + kk * 8 * LD);
    const float2 bb = *reinterpret_cast<const float2*>(&s.beta[ia]);
    uint32_t a0[4] = {tf32(M0[ia * LDS + ja]), tf32(M0[ia * LDS + jb]), tf32(M0[ib * LDS + ja]),
                      tf32(M0[ib * LDS + jb])};
    uint32_t a1[4] = {tf32(bb.x * M1[ia * LDS + ja]), tf32(bb.x * M1[ia * LDS + jb]), tf32(bb.y * M1[ib * LDS + ja]),
                      tf32(bb.y * M1[ib * LDS + jb])};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float qa = bf_lo(yq[nt]), qb = bf_hi(yq[nt]), ka = bf_lo(yk[nt]), kb = bf_hi(yk[nt]);
      if (VEC) {
        const int c = c0 + nt * 8 + g;
        const float ea = ex2(s.G[ia * LG + c] - mJ[nt]), eb = ex2(s.G[ib * LG + c] - mJ[nt]);
        qa *= ea;
        ka *= ea;
        qb *= eb;
        kb *= eb;
      }
      uint32_t b0[2] = {tf32(qa), tf32(qb)};
      uint32_t b1[2] = {tf32(ka), tf32(kb)};
      mma8(dst[nt], a0, b0);
      mma8(dst[nt], a1, b1);
    }
  }
  if (VEC)
    acc_foreach(acc, [&](int r, int col, float& x) {
      Z[col >> 3][(r >> 3) * 2 + (col & 1)] += x * ex2(s.G[mref * LG + c0 + col] - s.G[(j0b + r) * LG + c0 + col]);
    });
}

}  // namespace gdr
