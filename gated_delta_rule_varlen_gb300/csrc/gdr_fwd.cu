// gdr_fwd.cu -- forward kernel: the WY prep (the state walks are in gdr_walk.cu).
#include "gdr_chunk.cuh"
#include "gdr_kernels.h"
#include "gdr_tc.cuh"

namespace gdr {

// ---------------------------------------------------------------------------
// KDA prep (one CTA of 8 warps per (chunk, head); grouped GDN's scalar gate
// has the tensor-core prep k_prep_gdn below): gate cumsum, gated Gram
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
  constexpr int LDK = ChunkSmemB::LD, LG = ChunkSmemB::LG;
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
  // Each thread keeps two channels, d = 2 (tid % 64) and d + 1, in the pass
  // below; their gc_last is read before the pass overwrites the gate tile.
  const int dch = 2 * (tid & (DK / 2 - 1));
  const float2 glast = VEC ? *reinterpret_cast<const float2*>(&s.G[(CH - 1) * LG + dch])
                           : make_float2(s.gs[CH - 1], s.gs[CH - 1]);
  __syncthreads();  // At is stored (or unused) and every gc_last is read
  // v rows (async) into the At tile, free from here on (BF16 rows at the q/k
  // pitch take exactly its size).
  uint16_t* const Vt = reinterpret_cast<uint16_t*>(s.At);
  static_assert(sizeof(s.At) == CH * LDK * sizeof(uint16_t), "the v tile takes the At tile's place");
  for (int e = tid; e < CH * DK / 8; e += blockDim.x) {
    const int i = e >> 4, d8 = (e & 15) * 8;
    if (i < cd.len)
      cp_async16(&Vt[i * LDK + d8], a.v + ((size_t)(cd.tok0 + i) * a.HV + h) * DK + d8);
    else
      *reinterpret_cast<uint4*>(&Vt[i * LDK + d8]) = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_async_commit();
  // One elementwise pass: thread (channels d, d + 1, rows i0 .. i0 + 7) forms
  //   Kd = K exp(gc_last - gc)  one 16-byte piece of Kd^T per channel ([c][j],
  //                             the operand layout of the walk's state update),
  //   Qp = Q exp(gc)            one FP16 pair per row,
  //   beta K exp(gc)            the B operand of w, FP32, in place of gc,
  // and gamma = exp(gc_last) with the channels' first pieces.  Kd and Qp are
  // only ever MMA operands and their factors are <= 1: stored in FP16.
  for (int e = tid; e < DK * CH / 16; e += blockDim.x) {
    const int d = 2 * (e & (DK / 2 - 1)), i0 = 8 * (e >> 6);
    if (i0 == 0)
      *reinterpret_cast<float2*>(&a.gam[((size_t)chunk * a.HV + h) * DK + d]) = make_float2(ex2(glast.x), ex2(glast.y));
    __half* const qo = a.qp + qp_off(chunk, h, a.HV) + d;
    uint32_t p0[4], p1[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float kd0[2], kd1[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = i0 + 2 * q + u;
        const float2 gc = VEC ? *reinterpret_cast<const float2*>(&s.G[i * LG + d]) : make_float2(s.gs[i], s.gs[i]);
        const float2 kv = s.k2(i, d), qv = s.q2(i, d);
        const float rk = scaled ? s.rk[i] : 1.f, rq = scaled ? s.rq[i] : 1.f;
        kd0[u] = kv.x * rk * ex2(glast.x - gc.x);
        kd1[u] = kv.y * rk * ex2(glast.y - gc.y);
        const float gm0 = ex2(gc.x), gm1 = ex2(gc.y);
        *reinterpret_cast<__half2*>(&qo[i * DK]) = __floats2half2_rn(qv.x * rq * gm0, qv.y * rq * gm1);
        const float bk = s.beta[i] * rk;
        *reinterpret_cast<float2*>(&s.G[i * LG + d]) = make_float2(bk * kv.x * gm0, bk * kv.y * gm1);
      }
      const __half2 h0 = __floats2half2_rn(kd0[0], kd0[1]), h1 = __floats2half2_rn(kd1[0], kd1[1]);
      p0[q] = *reinterpret_cast<const uint32_t*>(&h0);
      p1[q] = *reinterpret_cast<const uint32_t*>(&h1);
    }
    __half* const ko = a.kd + kd_off(chunk, h, a.HV) + d * CH + i0;
    *reinterpret_cast<uint4*>(ko) = make_uint4(p0[0], p0[1], p0[2], p0[3]);
    *reinterpret_cast<uint4*>(ko + CH) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
  }
  cp_async_wait<0>();
  __syncthreads();
  // w (warps 0-3) and u (warps 4-7) = T B over rows j <= i.  Warp q of a
  // product takes channel half q % 2 of row blocks {3, 0} (q < 2) or {2, 1},
  // so that the four warps do equal work.  B of u, beta_j V_jc, is formed from
  // the BF16 v tile (in the At tile) as it is read: each k-step (rows j = 8 kk
  // .. 8 kk + 7) puts rows 8 kk + 2t and 8 kk + 2t + 1 in the k slots t and
  // t + 4 (the order within a step is free), so that the B fragments of four
  // n-tiles come from one transposing 8 x 8 matrix load of v, and each A
  // fragment row of T is one float2.  w reads its FP32 B tile (row pitch 136)
  // with the rows in the slots as they come.
  {
    const int prod = warp >> 2, q = warp & 3, c0 = 64 * (q & 1);
    const int Ia = (q >> 1) ? 2 : 3, Ib = 3 - Ia;
    const int lane = lane_id(), g = lane >> 2, t = lane & 3;
    __half* uo = a.u + tf_off(chunk, h, a.HV);
    __half* wo = a.w + w_off(chunk, h, a.HV);
    // This lane's row of the 8 x 8 matrices of v (n-tile lane / 8 of each group of four, row lane % 8).
    const uint16_t* const vrow = Vt + (lane & 7) * LDK + c0 + 8 * (lane >> 3);
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int I = pass ? Ib : Ia, i0 = 16 * I;
      float acc[8][4];
      zero_acc(acc);
#pragma unroll 2
      for (int kk = 0; kk < 2 * I + 2; ++kk) {
        if (prod) {
          const int j0 = kk * 8 + 2 * t;
          const float2 ta = *reinterpret_cast<const float2*>(&s.T[(i0 + g) * LDS + j0]);
          const float2 tb = *reinterpret_cast<const float2*>(&s.T[(i0 + g + 8) * LDS + j0]);
          const uint32_t af[4] = {tf32(ta.x), tf32(tb.x), tf32(ta.y), tf32(tb.y)};
          uint32_t y[2][4];
          ldsm_x4_trans(y[0], vrow + kk * 8 * LDK);
          ldsm_x4_trans(y[1], vrow + kk * 8 * LDK + 32);
          const float2 bb = *reinterpret_cast<const float2*>(&s.beta[j0]);
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) {
            const uint32_t yv = y[nt >> 2][nt & 3];
            uint32_t b[2] = {tf32(bb.x * bf_lo(yv)), tf32(bb.y * bf_hi(yv))};
            mma8(acc[nt], af, b);
          }
        } else {
          const int ja = kk * 8 + t, jb = ja + 4;
          const uint32_t af[4] = {tf32(s.T[(i0 + g) * LDS + ja]), tf32(s.T[(i0 + g + 8) * LDS + ja]),
                                  tf32(s.T[(i0 + g) * LDS + jb]), tf32(s.T[(i0 + g + 8) * LDS + jb])};
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) {
            const int c = c0 + nt * 8 + g;
            uint32_t b[2] = {tf32(s.G[ja * LG + c]), tf32(s.G[jb * LG + c])};
            mma8(acc[nt], af, b);
          }
        }
      }
      {  // rows i0 + g (+8), channel pairs c0 + 8 nt + 2 t: FP16 pairs
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int row = i0 + g + 8 * hr, c = c0 + nt * 8 + 2 * t;
            const __half2 p = __floats2half2_rn(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
            if (prod)
              *reinterpret_cast<__half2*>(&uo[row * LDF + c]) = p;
            else
              *reinterpret_cast<__half2*>(&wo[row * DK + c]) = p;
          }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Prep of grouped GDN on the tensor cores: one CTA of 8 warps per (chunk, Q/K
// head), the value heads of the group one after another.  With a scalar gate
// the gated Gram matrices are the raw products times a decay mask,
//   At[i][j]  = (K K^T)[i][j] exp(gc_i - gc_j)   (j <  i),
//   Aqk[i][j] = (Q K^T)[i][j] exp(gc_i - gc_j)   (j <= i),
// so [K K^T ; Q K^T] is one tcgen05.mma series (kind::f16: M = 128 rows
// [K ; Q], N = 64, K = 128 channels; exact products of the BF16 inputs, FP32
// accumulators in tensor memory) that every value head of the Q/K head
// shares.  Per value head: the gate cumsum, the masks (read from tensor
// memory), the inverse on the CUDA cores, then
//   w = (T diag(beta Gamma)) K,   u = (T diag(beta)) V
// as two more series (M = 64, N = 128, K = 64 tokens): A is the FP32 matrix
// split into a BF16 pair hi + lo (two MMAs per step), B the K or V tile as
// TMA brought it (a 128-byte-swizzled [token][channel] tile read MN-major is
// the B operand with the tokens as its K index).  With in-kernel L2
// normalization the row scales enter in FP32: the masks take r_i r_j, the A
// operand of w takes r_k.  Outputs as the per-value-head prep writes them:
// w, u, Q Gamma, Kd^T, Aqk, gamma and (saving forward) At, T.
// The "prep program" of PR #8638 "perf(cake_gdn_kcp): ... graph-replay
// checkpoint recompute hands its tapes to the backward", with the grouping
// of value heads by Q/K head of PR #7723 "perf(cake_gdn): prefetch offset
// adjoint walk, default LPT segment plan" (opening description).
// ---------------------------------------------------------------------------
struct __align__(16) PrepGdnSmem {
  uint16_t KQ[2 * 2 * CH * 64];  // 2 channel blocks x [k rows 0..63 ; q rows 64..127] x 64 channels (SW128)
  uint16_t V[2 * CH * 64];       // v of one value head: 2 channel blocks x 64 rows (SW128)
  uint16_t A[2][CH * 64];        // A of w, then of u: BF16 hi, lo (K-major SW128, 64 rows x 64 tokens)
  float At[CH * LDS];
  float T[CH * LDS];
  float tmp[6 * 128];
  float gin[2][CH], bin[2][CH];  // g and beta of a value head, one ahead (cp.async)
  float gs[CH], beta[CH], rq[CH], rk[CH];
  float bw[CH];  // beta_j Gamma_j r_k,j
  float gm[CH];  // Gamma_i = exp(gc_i)
  float ed[CH];  // exp(gc_last - gc_i)
  uint64_t bar_qk, bar_v, bar_g, bar_m;
  uint32_t tmem;
};
constexpr uint32_t PREP_TC_COLS = 256;       // Gram [0, 64); w, then u, [128, 256)
constexpr uint32_t KQ_BLOCK = 2 * CH * 128;  // bytes of one channel block of [k ; q]
constexpr uint32_t V_BLOCK = CH * 128;       // bytes of one channel block of v

// Byte offset of BF16 element (row r, channel c) in a 128-byte-swizzled tile
// of channel blocks `block` bytes apart.
__device__ __forceinline__ uint32_t sw_elem(int r, int c, uint32_t block) {
  const int cc = c & 63;
  return (uint32_t)(c >> 6) * block + (uint32_t)r * 128 + ((((cc >> 3) ^ (r & 7)) << 4) | ((cc & 7) << 1));
}

// One 4-byte asynchronous copy global -> shared.
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(gmem));
}

// A operand T diag(f) (rows i, tokens j; T lower triangular) as BF16 hi + lo
// in the K-major 128-byte-swizzled layout.  Item (row i, 8-token piece kc),
// the row fastest: a warp's lanes take 32 consecutive rows of one piece, so
// the two float4 reads of T per item fall on distinct banks, the eight
// factors f are one broadcast, and the swizzled 16-byte stores are
// conflict-free.
__device__ __forceinline__ void build_a(PrepGdnSmem& s, const float* __restrict__ f) {
  for (int e = threadIdx.x; e < CH * 8; e += blockDim.x) {
    const int i = e & (CH - 1), kc = e >> 6;
    const float4 t0 = *reinterpret_cast<const float4*>(&s.T[i * LDS + 8 * kc]);
    const float4 t1 = *reinterpret_cast<const float4*>(&s.T[i * LDS + 8 * kc + 4]);
    const float4 f0 = *reinterpret_cast<const float4*>(&f[8 * kc]);
    const float4 f1 = *reinterpret_cast<const float4*>(&f[8 * kc + 4]);
    const float x[8] = {t0.x * f0.x, t0.y * f0.y, t0.z * f0.z, t0.w * f0.w,
                        t1.x * f1.x, t1.y * f1.y, t1.z * f1.z, t1.w * f1.w};
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float x0 = x[2 * p], x1 = x[2 * p + 1];
      const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
      const __nv_bfloat16 l0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
      const __nv_bfloat16 l1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
      hi[p] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      lo[p] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    const uint32_t off = tc::sw128_bf16_piece(i, kc, CH);
    *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(s.A[0]) + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(s.A[1]) + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// The M = 64 accumulator at TMEM column 128 (w or u) -> FP16 rows of `out`,
// `ld` elements apart.  Warp (quadrant, half): rows 16 quad .., channels 64 half ..
__device__ __forceinline__ void drain_wu(uint32_t tmem, __half* __restrict__ out, int ld) {
  const int warp = threadIdx.x >> 5, lane = lane_id();
  const int quad = warp & 3, hf = warp >> 2, g = lane >> 2, u2 = (lane & 3) * 2;
  const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16) + 128 + 64 * hf;
#pragma unroll 1
  for (int cb = 0; cb < 64; cb += 16) {
    uint32_t rr[8];
    tc::tmem_ld16x256b_x2(tq + cb, rr);
    tc::tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = 16 * quad + g + 8 * hr, c = 64 * hf + cb + 8 * q + u2;
        const float x0 = __uint_as_float(rr[4 * q + 2 * hr]), x1 = __uint_as_float(rr[4 * q + 2 * hr + 1]);
        *reinterpret_cast<__half2*>(&out[row * ld + c]) = __floats2half2_rn(x0, x1);
      }
  }
}

__global__ void __launch_bounds__(256, 2) k_prep_gdn(const __grid_constant__ PrepTcArgs ta) {
  const PrepArgs& a = ta.p;
  extern __shared__ unsigned char smraw[];
  PrepGdnSmem& s = *reinterpret_cast<PrepGdnSmem*>(tc::align1024(smraw));
  const int chunk = a.chunk_base + blockIdx.x, hq = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int G = a.HV / a.Hqk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = lane_id();
  const bool scaled = a.rq != nullptr;
  const float* beta = static_cast<const float*>(a.beta);
  unsigned char* kq = reinterpret_cast<unsigned char*>(s.KQ);
  unsigned char* vt = reinterpret_cast<unsigned char*>(s.V);
  if (tid == 0) {
    tc::mbar_init(&s.bar_qk, 1);
    tc::mbar_init(&s.bar_v, 1);
    tc::mbar_init(&s.bar_g, 1);
    tc::mbar_init(&s.bar_m, 1);
    tc::mbar_fence_init();
    tc::mbar_arrive_expect_tx(&s.bar_qk, 2 * KQ_BLOCK);
    for (int kb = 0; kb < 2; ++kb) {
      tc::tma_load_3d(kq + kb * KQ_BLOCK, &ta.k_map, 64 * kb, hq, cd.tok0, &s.bar_qk);
      tc::tma_load_3d(kq + kb * KQ_BLOCK + CH * 128, &ta.q_map, 64 * kb, hq, cd.tok0, &s.bar_qk);
    }
    tc::mbar_arrive_expect_tx(&s.bar_v, 2 * V_BLOCK);
    for (int kb = 0; kb < 2; ++kb) tc::tma_load_3d(vt + kb * V_BLOCK, &ta.v_map, 64 * kb, hq * G, cd.tok0, &s.bar_v);
  }
  if (warp == 0) {
    tc::tmem_alloc(&s.tmem, PREP_TC_COLS);
    tc::tmem_relinquish();
  }
  // Gate and beta of value head h (rows past the chunk: zero) into buffer b.
  auto fetch_gb = [&](int h, int b) {
    if (tid < CH) {
      if (tid < cd.len) {
        const size_t idx = (size_t)(cd.tok0 + tid) * a.HV + h;
        cp_async4(&s.gin[b][tid], a.g + idx);
        cp_async4(&s.bin[b][tid], beta + idx);
      } else {
        s.gin[b][tid] = 0.f;
        s.bin[b][tid] = 0.f;
      }
      cp_async_commit();
    }
  };
  fetch_gb(hq * G, 0);
  if (tid < CH) {
    const size_t row = (size_t)(cd.tok0 + min(tid, max(cd.len - 1, 0))) * a.Hqk + hq;
    s.rq[tid] = scaled ? a.rq[row] : 1.f;
    s.rk[tid] = scaled ? a.rk[row] : 1.f;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s.tmem;
  // Rows past the chunk's tokens (the next document's, or zero fill past T) -> zero.
  bool ok = tc::mbar_wait(&s.bar_qk, 0);
  if (ok && cd.len < CH)
    for (int e = tid; e < (CH - cd.len) * 32; e += 256) {  // row, {k, q}, channel block, 16-byte piece
      const int p = e & 7, kb = (e >> 3) & 1, isq = (e >> 4) & 1, i = cd.len + (e >> 5);
      *reinterpret_cast<uint4*>(kq + kb * KQ_BLOCK + (isq * CH + i) * 128 + p * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
  tc::fence_proxy_async();
  ok = __syncthreads_and(ok);
  bool g_issued = false;
  if (ok && tid == 0) {
    tc::tc_fence_after();
    const uint64_t d = tc::desc_k_sw128(kq);
    constexpr uint32_t idg = tc::idesc_bf16(2 * CH, CH);
#pragma unroll
    for (int k = 0; k < 8; ++k) tc::mma_bf16(tmem, tc::kstep32(d, k, 2 * CH), tc::kstep32(d, k, 2 * CH), idg, k > 0);
    tc::mma_commit(&s.bar_g);
    g_issued = true;
  }
  // What a timed-out CTA still waits for (the same counts in every thread).
  int v_issued = 1, v_waited = 0, m_issued = 0, m_waited = 0;
  constexpr uint32_t idw = tc::idesc_bf16(CH, DK) | tc::kIdescTransposeB;  // B MN-major (tokens = K)
  for (int r = 0; r < G && ok; ++r) {
    const int h = hq * G + r, pb = r & 1;
    if (r + 1 < G) fetch_gb(h + 1, pb ^ 1);
    // Gate cumsum (base 2), beta and the per-row factors of value head h.
    if (tid < CH) {
      if (r + 1 < G)
        cp_async_wait<1>();
      else
        cp_async_wait<0>();
      s.beta[tid] = s.bin[pb][tid];
      float x = s.gin[pb][tid] * LOG2E;
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
    if (tid < CH) {
      const float x = s.gs[tid];
      s.gm[tid] = ex2(x);
      s.ed[tid] = ex2(s.gs[CH - 1] - x);
      s.bw[tid] = s.beta[tid] * s.gm[tid] * s.rk[tid];
    }
    ok = __syncthreads_and(tc::mbar_wait(&s.bar_g, 0));  // the Gram (completes once)
    tc::tc_fence_after();
    if (!ok) break;
    {  // Masks.  Warp (lane quadrant qd, half hf): rows 32 (qd & 1) + lane of K K^T (qd < 2)
       // or Q K^T (qd >= 2), columns j = 32 hf .. 32 hf + 31.
      const int qd = warp & 3, hf = warp >> 2, i = 32 * (qd & 1) + lane;
      const bool isq = qd >= 2;
      const float gi = s.gs[i], ri = isq ? s.rq[i] : s.rk[i];
      __half* aq_row = a.aqk + aqk_off(chunk, h, a.HV) + i * CH;
      float* at_row = s.At + i * LDS;
#pragma unroll 1
      for (int j0 = 32 * hf; j0 < 32 * hf + 32; j0 += 16) {
        uint32_t v[16];
        tc::tmem_ld16(tmem + ((uint32_t)(32 * qd) << 16) + j0, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j4 = 0; j4 < 16; j4 += 4) {
          float o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int j = j0 + j4 + q;
            const bool keep = isq ? j <= i : j < i;
            const float x = ((__uint_as_float(v[j4 + q]) * ex2(gi - s.gs[j])) * ri) * s.rk[j];
            o[q] = keep ? x : 0.f;
          }
          if (isq) {
            const __half2 p0 = __floats2half2_rn(o[0], o[1]), p1 = __floats2half2_rn(o[2], o[3]);
            *reinterpret_cast<uint2*>(aq_row + j0 + j4) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1));
          } else {
            *reinterpret_cast<float4*>(at_row + j0 + j4) = make_float4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    }
    __syncthreads();
    invert_tiles(s.At, s.T, s.beta, s.tmp);
    // w = (T diag(beta Gamma r_k)) K.
    build_a(s, s.bw);
    tc::fence_proxy_async();
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc::tc_fence_after();
#pragma unroll
      for (int hl = 0; hl < 2; ++hl) {
        const uint64_t ad = tc::desc_k_sw128(s.A[hl]);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + 128, tc::kstep32(ad, ks, CH), tc::desc_mn_sw128(kq + ks * 16 * 128, KQ_BLOCK, 1024), idw,
                       (hl | ks) != 0);
      }
      tc::mma_commit(&s.bar_m);
    }
    ++m_issued;
    // While it runs: Q Gamma and Kd^T.
    for (int e = tid; e < CH * DK / 4; e += 256) {  // four channels per thread, one 8-byte store
      const int i = e >> 5, d = (e & 31) * 4;
      const uint2 raw = *reinterpret_cast<const uint2*>(kq + sw_elem(CH + i, d, KQ_BLOCK));
      const float f = s.rq[i] * s.gm[i];
      const float x0 = __uint_as_float(raw.x << 16), x1 = __uint_as_float(raw.x & 0xffff0000u);
      const float x2 = __uint_as_float(raw.y << 16), x3 = __uint_as_float(raw.y & 0xffff0000u);
      const __half2 p0 = __floats2half2_rn(x0 * f, x1 * f), p1 = __floats2half2_rn(x2 * f, x3 * f);
      *reinterpret_cast<uint2*>(&a.qp[qp_off(chunk, h, a.HV) + i * DK + d]) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1));
    }
    for (int e = tid; e < DK * CH / 8; e += 256) {  // Kd^T [c][j]: thread (channel d, rows i0 .. i0 + 7), 16 bytes
      const int d = e & (DK - 1), i0 = 8 * (e >> 7);
      uint32_t p[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + 2 * q;
        const uint16_t r0 = *reinterpret_cast<const uint16_t*>(kq + sw_elem(i, d, KQ_BLOCK));
        const uint16_t r1 = *reinterpret_cast<const uint16_t*>(kq + sw_elem(i + 1, d, KQ_BLOCK));
        const __half2 hv = __floats2half2_rn(bfbits2f(r0) * s.rk[i] * s.ed[i], bfbits2f(r1) * s.rk[i + 1] * s.ed[i + 1]);
        p[q] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      *reinterpret_cast<uint4*>(&a.kd[kd_off(chunk, h, a.HV) + d * CH + i0]) = make_uint4(p[0], p[1], p[2], p[3]);
    }
    ok = __syncthreads_and(tc::mbar_wait(&s.bar_m, 0));
    ++m_waited;
    tc::tc_fence_after();
    if (!ok) break;
    drain_wu(tmem, a.w + w_off(chunk, h, a.HV), DK);
    tc::tc_fence_before();
    __syncthreads();
    // u = (T diag(beta)) V.
    build_a(s, s.beta);
    bool okv = tc::mbar_wait(&s.bar_v, r & 1);
    ++v_waited;
    if (okv && cd.len < CH)
      for (int e = tid; e < (CH - cd.len) * 16; e += 256) {  // row, channel block, 16-byte piece
        const int p = e & 7, kb = (e >> 3) & 1, i = cd.len + (e >> 4);
        *reinterpret_cast<uint4*>(vt + kb * V_BLOCK + i * 128 + p * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    tc::fence_proxy_async();
    ok = __syncthreads_and(okv);
    if (!ok) break;
    if (tid == 0) {
      tc::tc_fence_after();
#pragma unroll
      for (int hl = 0; hl < 2; ++hl) {
        const uint64_t ad = tc::desc_k_sw128(s.A[hl]);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + 128, tc::kstep32(ad, ks, CH), tc::desc_mn_sw128(vt + ks * 16 * 128, V_BLOCK, 1024), idw,
                       (hl | ks) != 0);
      }
      tc::mma_commit(&s.bar_m);
    }
    ++m_issued;
    // While it runs: gamma, and At, T for the backward.
    if (tid < DK) a.gam[((size_t)chunk * a.HV + h) * DK + tid] = s.gm[CH - 1];
    if (a.amat) {
      const size_t qo = ts_off(chunk, h, a.HV);
      for (int e = tid; e < CH * CH / 4; e += 256) {
        const int i = e >> 4, j4 = (e & 15) * 4;
        *reinterpret_cast<float4*>(&a.amat[qo + i * LDS + j4]) = *reinterpret_cast<const float4*>(&s.At[i * LDS + j4]);
        *reinterpret_cast<float4*>(&a.tmat[qo + i * LDS + j4]) = *reinterpret_cast<const float4*>(&s.T[i * LDS + j4]);
      }
    }
    ok = __syncthreads_and(tc::mbar_wait(&s.bar_m, 1));
    ++m_waited;
    tc::tc_fence_after();
    if (!ok) break;
    if (r + 1 < G) {  // the v tile is free: the next value head's
      if (tid == 0) {
        tc::mbar_arrive_expect_tx(&s.bar_v, 2 * V_BLOCK);
        for (int kb = 0; kb < 2; ++kb) tc::tma_load_3d(vt + kb * V_BLOCK, &ta.v_map, 64 * kb, h + 1, cd.tok0, &s.bar_v);
      }
      ++v_issued;
    }
    drain_wu(tmem, a.u + tf_off(chunk, h, a.HV), LDF);
    tc::tc_fence_before();
    __syncthreads();
  }
  if (tid < CH) cp_async_wait<0>();
  if (!ok && tid == 0) {
    // A wait ran out: record it and let the copies and products in flight finish.
    atomicExch(ta.err, 9);
    tc::mbar_wait(&s.bar_qk, 0);
    if (g_issued) tc::mbar_wait(&s.bar_g, 0);
    if (v_waited < v_issued) tc::mbar_wait(&s.bar_v, v_waited & 1);
    if (m_waited < m_issued) tc::mbar_wait(&s.bar_m, m_waited & 1);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, PREP_TC_COLS);
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
cudaError_t launch_prep(const PrepArgs& a, int nchunks, cudaStream_t st) {
  if (nchunks == 0) return cudaSuccess;
  const size_t sm = sizeof(ChunkSmemB);
  cudaFuncSetAttribute(k_prep<true, __nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  k_prep<true, __nv_bfloat16><<<dim3(nchunks, a.HV), 256, sm, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prep_gdn(const PrepTcArgs& a, int nchunks, cudaStream_t st) {
  if (nchunks == 0) return cudaSuccess;
  const size_t sm = sizeof(PrepGdnSmem) + 1024;
  cudaFuncSetAttribute(k_prep_gdn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  k_prep_gdn<<<dim3(nchunks, a.p.Hqk), 256, sm, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdr
