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
#include "gdr_tc.cuh"

namespace gdr {

// ---------------------------------------------------------------------------
// State-side products on the tensor cores (one CTA of 8 warps per (chunk,
// value head)):
//   dqs = scale dO S0^T,  dw = -dDelta S0^T,  dKd = Delta dS^T,
//   dAqk = scale tril(dO Delta^T),  dgam[c] = sum_v dS[c][v] S0[c][v].
// tcgen05.mma kind::f16 (BF16 operands, FP32 accumulators in TMEM, M = 64
// tokens).  dO and the two state tapes are BF16 already; Delta and dDelta are
// FP32 and enter as a BF16 pair hi + lo (hi = bf16(x), lo = bf16(x - hi),
// about 16 significant bits), so each of their products is two MMAs.  Both
// state tapes are stored chunk-major (element (v, c) of a chunk's tile at
// ((c / 8) * 128 + v) * 8 + c % 8, as the walks write them) and arrive as one
// bulk copy each; that layout is the canonical no-swizzle MN-major operand
// layout (8 channels x 8 value columns per 128-byte core matrix), so they are
// the B operands (N = channel c, K = value column v) as they are.
// ---------------------------------------------------------------------------
struct GradStateSmem {
  uint16_t Tp[DK * DK];      // B (MN-major, no swizzle): the S0 tape tile, then the dS tape tile
  uint16_t dO[2 * CH * 64];  // A: dO [i][v]
  uint16_t Hi[2 * CH * 64];  // dDelta hi [i][v] (A of dw), then Delta hi (A of dKd, B of dAqk)
  uint16_t Lo[2 * CH * 64];  // the lo parts
  uint64_t bar_t1, bar_t2, bar_m1, bar_m2;
  uint32_t tmem;
};

// FP32 rows of a [64][128] tile (pitch ld) -> BF16 hi / lo pairs in the
// swizzled K-major A layout: task e = row (e / 16), 16-byte piece e % 16;
// x holds the 8 values of each of the thread's 4 tasks.
__device__ __forceinline__ void load_hilo_rows(const float* __restrict__ src, int ld, float4 (&x)[4][2]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = threadIdx.x + 256 * q;
    const float* p = src + (size_t)(e >> 4) * ld + (e & 15) * 8;
    x[q][0] = __ldg(reinterpret_cast<const float4*>(p));
    x[q][1] = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
}
__device__ __forceinline__ void store_hilo_rows(const float4 (&x)[4][2], uint16_t* hi_t, uint16_t* lo_t) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = threadIdx.x + 256 * q;
    const float f[8] = {x[q][0].x, x[q][0].y, x[q][0].z, x[q][0].w, x[q][1].x, x[q][1].y, x[q][1].z, x[q][1].w};
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(f[2 * p]), h1 = __float2bfloat16_rn(f[2 * p + 1]);
      const __nv_bfloat16 l0 = __float2bfloat16_rn(f[2 * p] - __bfloat162float(h0));
      const __nv_bfloat16 l1 = __float2bfloat16_rn(f[2 * p + 1] - __bfloat162float(h1));
      hi[p] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      lo[p] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    const uint32_t off = tc::sw128_bf16_piece(e >> 4, e & 15, CH);
    *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(hi_t) + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(lo_t) + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// Two phases in one CTA, so that two CTAs fit on an SM (256 TMEM columns,
// ~80 KB of shared memory) and one CTA's copies overlap the other's products:
//   1. dqs = scale dO S0^T (TMEM 0..127), dw = -dDelta S0^T (128..255);
//   2. (the dS tape into the S0 tape's place, Delta's pairs into dDelta's)
//      dKd = Delta dS^T (0..127), dAqk = scale tril(dO Delta^T) (128..191);
// and dgam from the dS tile and the S0 tape read again (from L2).
__global__ void __launch_bounds__(256, 2) k_grad_state(const __grid_constant__ GradStateArgs a) {
  extern __shared__ unsigned char smraw[];
  GradStateSmem& s = *reinterpret_cast<GradStateSmem*>(tc::align1024(smraw));
  const int chunk = a.chunk_base + blockIdx.x, h = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int tid = threadIdx.x, warp = tid >> 5, lane = lane_id();
  const size_t toff = tile_off(chunk, h, a.HV);
  constexpr uint32_t TCOLS = 256;
  if (tid == 0) {
    tc::mbar_init(&s.bar_t1, 1);
    tc::mbar_init(&s.bar_t2, 1);
    tc::mbar_init(&s.bar_m1, 1);
    tc::mbar_init(&s.bar_m2, 1);
    tc::mbar_fence_init();
    tc::mbar_arrive_expect_tx(&s.bar_t1, DK * DK * 2);
    tc::bulk_load(s.Tp, a.tape + state_off(chunk, h, a.HV), DK * DK * 2, &s.bar_t1);
  }
  if (warp == 0) {
    tc::tmem_alloc(&s.tmem, TCOLS);
    tc::tmem_relinquish();
  }
  unsigned char* sdO = reinterpret_cast<unsigned char*>(s.dO);
  // dO rows (zero beyond the chunk) into the swizzled A tile.
  for (int e = tid; e < CH * 16; e += 256) {
    const int i = e >> 4, kc = e & 15;
    void* dst = sdO + tc::sw128_bf16_piece(i, kc, CH);
    if (i < cd.len)
      cp_async16(dst, &a.dout[((size_t)(cd.tok0 + i) * a.HV + h) * DK + kc * 8]);
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_async_commit();
  float4 x[4][2];
  load_hilo_rows(a.ddelta + tf_off(chunk, h, a.HV), LDF, x);
  store_hilo_rows(x, s.Hi, s.Lo);
  load_hilo_rows(a.delta + toff, DK, x);  // Delta, for the second phase: its latency hides behind the first
  cp_async_wait<0>();
  tc::fence_proxy_async();
  bool ok = tc::mbar_wait(&s.bar_t1, 0);
  tc::tc_fence_before();
  ok = __syncthreads_and(ok);
  tc::tc_fence_after();
  const uint32_t tmem = s.tmem;
  constexpr uint32_t id64 = tc::idesc_bf16(CH, CH);
  constexpr uint32_t id128t = tc::idesc_bf16(CH, DK) | tc::kIdescTransposeB;  // B MN-major
  // K step k (16 value columns v: two core matrices of 8 v, 128 bytes apart) of
  // a chunk-major state tile; 8-channel groups are 128 x 16 bytes apart.
  auto bmn = [](const uint16_t* tile, int k) { return tc::desc_mn_none(tile + k * 16 * 8, 128, DK * 16); };
  if (ok && tid == 0) {
    const uint64_t aO = tc::desc_k_sw128(s.dO);
    const uint64_t aH = tc::desc_k_sw128(s.Hi), aL = tc::desc_k_sw128(s.Lo);
#pragma unroll
    for (int k = 0; k < 8; ++k) tc::mma_bf16(tmem, tc::kstep32(aO, k, CH), bmn(s.Tp, k), id128t, k > 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) tc::mma_bf16(tmem + 128, tc::kstep32(aH, k, CH), bmn(s.Tp, k), id128t, k > 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) tc::mma_bf16(tmem + 128, tc::kstep32(aL, k, CH), bmn(s.Tp, k), id128t, 1);
    tc::mma_commit(&s.bar_m1);
  }
  // Epilogue helpers: warp w reads the rows of TMEM lane quadrant w % 4 (tokens
  // 16 (w % 4) ..) and half w / 4 of the columns.
  const int quad = warp & 3, hf = warp >> 2, g = lane >> 2, u2 = (lane & 3) * 2;
  const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);
  auto drain = [&](uint32_t col0, int ncols, auto&& store) {  // ncols multiple of 16
    for (int cb = 0; cb < ncols; cb += 16) {
      uint32_t r[8];
      tc::tmem_ld16x256b_x2(tq + col0 + cb, r);
      tc::tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr)
          store(16 * quad + g + 8 * hr, cb + 8 * q + u2, __uint_as_float(r[4 * q + 2 * hr]),
                __uint_as_float(r[4 * q + 2 * hr + 1]));
    }
  };
  const bool ok1 = __syncthreads_and(ok && tc::mbar_wait(&s.bar_m1, 0));  // uniform: the loads below are warp-wide
  tc::tc_fence_after();
  if (ok1 && tid == 0) {  // the S0 tape's products are done: the dS tape into its place
    tc::mbar_arrive_expect_tx(&s.bar_t2, DK * DK * 2);
    tc::bulk_load(s.Tp, a.dstape + state_off(chunk, h, a.HV), DK * DK * 2, &s.bar_t2);
  }
  if (ok1) {
    store_hilo_rows(x, s.Hi, s.Lo);  // Delta hi / lo in dDelta's place
    const int c0 = 64 * hf;
    drain(c0, 64, [&](int i, int c, float x0, float x1) {
      *reinterpret_cast<float2*>(&a.dqs[toff + i * DK + c0 + c]) = make_float2(a.scale * x0, a.scale * x1);
    });
    drain(128 + c0, 64, [&](int i, int c, float x0, float x1) {
      *reinterpret_cast<float2*>(&a.dw[tf_off(chunk, h, a.HV) + i * LDF + c0 + c]) = make_float2(-x0, -x1);
    });
  }
  tc::fence_proxy_async();
  tc::tc_fence_before();
  const bool ok2 = __syncthreads_and(ok1 && tc::mbar_wait(&s.bar_t2, 0));
  tc::tc_fence_after();
  if (ok2 && tid == 0) {
    const uint64_t aO = tc::desc_k_sw128(s.dO);
    const uint64_t aH = tc::desc_k_sw128(s.Hi), aL = tc::desc_k_sw128(s.Lo);
#pragma unroll
    for (int k = 0; k < 8; ++k) tc::mma_bf16(tmem, tc::kstep32(aH, k, CH), bmn(s.Tp, k), id128t, k > 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) tc::mma_bf16(tmem, tc::kstep32(aL, k, CH), bmn(s.Tp, k), id128t, 1);
#pragma unroll
    for (int k = 0; k < 8; ++k) tc::mma_bf16(tmem + 128, tc::kstep32(aO, k, CH), tc::kstep32(aH, k, CH), id64, k > 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) tc::mma_bf16(tmem + 128, tc::kstep32(aO, k, CH), tc::kstep32(aL, k, CH), id64, 1);
    tc::mma_commit(&s.bar_m2);
  }
  if (ok2) {  // dgam[c] = sum_v S0[c][v] dS[c][v]: thread (q, vg) sums channels 8 q .. 8 q + 7 over
              // value columns vg, vg + 16, ..; the 16 partial sums of a channel group are then
              // added within the half warp in a fixed order.  S0 from the tape in memory.
    const int q = tid >> 4, vg = tid & 15;
    const uint4* p0 = reinterpret_cast<const uint4*>(a.tape + state_off(chunk, h, a.HV)) + q * DK;
    const uint4* p1 = reinterpret_cast<const uint4*>(s.Tp) + q * DK;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint4 xs4 = __ldg(p0 + vg + 16 * r), y = p1[vg + 16 * r];
      const uint32_t xs[4] = {xs4.x, xs4.y, xs4.z, xs4.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        acc[2 * p] += __uint_as_float(xs[p] << 16) * __uint_as_float(ys[p] << 16);
        acc[2 * p + 1] += __uint_as_float(xs[p] & 0xffff0000u) * __uint_as_float(ys[p] & 0xffff0000u);
      }
    }
#pragma unroll
    for (int off = 1; off < 16; off <<= 1)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
    if (vg == 0) {
#pragma unroll
      for (int e = 0; e < 8; ++e) a.dgam[((size_t)chunk * a.HV + h) * DK + 8 * q + e] = acc[e];
    }
  }
  const bool ok3 = __syncthreads_and(ok2 && tc::mbar_wait(&s.bar_m2, 0));
  tc::tc_fence_after();
  if (ok3) {
    const int c0 = 64 * hf;
    drain(c0, 64, [&](int i, int c, float x0, float x1) {
      *reinterpret_cast<float2*>(&a.dkd[toff + i * DK + c0 + c]) = make_float2(x0, x1);
    });
    float* daqk = a.daqk + ts_off(chunk, h, a.HV);
    const int j0 = 32 * hf;
    drain(128 + j0, 32, [&](int i, int c, float x0, float x1) {
      const int j = j0 + c;
      *reinterpret_cast<float2*>(&daqk[i * LDS + j]) =
          make_float2(j <= i ? a.scale * x0 : 0.f, j + 1 <= i ? a.scale * x1 : 0.f);
    });
  }
  if (tid == 0 && !ok3) {
    // A wait ran out: record it and let the copies and products in flight finish.
    atomicExch(a.err, 6);
    tc::mbar_wait(&s.bar_t1, 0);
    if (ok) tc::mbar_wait(&s.bar_m1, 0);
    if (ok1) tc::mbar_wait(&s.bar_t2, 0);
    if (ok2) tc::mbar_wait(&s.bar_m2, 0);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TCOLS);
}

// ---------------------------------------------------------------------------
// Chunk-local gradients (one CTA per (chunk, value head)).  Warp I owns rows
// 16I..16I+15 of every per-row result; dk and the gate adjoint accumulate in
// registers, dg is the reverse chunk-local cumsum of dgc.  The
// "fused gradient" / "gate epilogue" stages named on PR #8218.
// ---------------------------------------------------------------------------
constexpr int GRAD_WARPS = 16;   // 4 row blocks x 4 channel quarters
constexpr int GRAD_NT = 4;       // 8-channel n-tiles per warp (32 channels)

struct GradSmem {
  ChunkSmemB c;       // its At tile holds w (FP16 rows LDF elements apart) instead
  float uh[CH * LDS];  // u: FP16 rows LDF elements apart (the same bytes)
  float dK[CH * LDF];  // staging: dw, then the forward's At and dAqk
  float dG[CH * LDF];  // staging: dDelta, then the gate adjoint dgc
  float dbeta[5][CH];  // per channel quarter (X.Kp + Y.V), and sum_j dA_ij At_ij
  float col[4 * DK];
  float rowsum[CH];
  uint64_t bar_ld, bar_w, bar_u;
};

// 16 warps: warp w owns channels 32 qc .. +31 (qc = w / 4) and rows 16 I ..
// +15 (I = (w + qc) % 4) of every per-row result, held in registers in the
// m16n8 accumulator layout (thread: rows i0 + g and i0 + g + 8, channel pairs
// c0 + 8 nt + 2 t).  Warp w issues from the SM sub-partition w % 4, so each
// sub-partition holds one warp of every row block and the triangular products
// (whose work grows or shrinks with I) split evenly over the four.  The one
// product that contracts over channels (dA) is summed over the four channel
// quarters in four ordered passes.
template <bool VEC, typename BetaT>
__global__ void __launch_bounds__(GRAD_WARPS * 32, 1) k_grad(GradArgs a) {
  constexpr int NT = GRAD_NT;
  constexpr int NTH = GRAD_WARPS * 32;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  GradSmem& sg = *reinterpret_cast<GradSmem*>(smem_raw);
  ChunkSmemB& s = sg.c;
  const int chunk = a.chunk_base + blockIdx.x, h = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int hq = h / (a.HV / a.Hqk);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int qc = warp >> 2, I = (warp + qc) & 3, i0 = 16 * I, c0 = 8 * NT * qc;
  const int lane = lane_id(), g = lane >> 2, t = lane & 3;
  const size_t toff = tile_off(chunk, h, a.HV);
  const size_t fo = tf_off(chunk, h, a.HV), so = ts_off(chunk, h, a.HV);
  // Everything the first products read, issued at once.  Whole tiles, stored
  // with these shared pitches, by one bulk copy each: the forward's T, dw and
  // dDelta (the operands of X and Y, waited for first), then u (FP16, a B
  // operand of dA, on a barrier of its own).  w (dense FP16 rows) by cp.async
  // into the At tile with u's pitch; the forward's At and dAqk follow once X
  // and Y have freed the dw staging tile.
  if (tid == 0) {
    tc::mbar_init(&sg.bar_ld, 1);
    tc::mbar_init(&sg.bar_w, 1);
    tc::mbar_init(&sg.bar_u, 1);
    tc::mbar_fence_init();
    tc::mbar_arrive_expect_tx(&sg.bar_ld, (2 * CH * LDF + CH * LDS) * 4);
    tc::bulk_load(s.T, &a.tmat[so], CH * LDS * 4, &sg.bar_ld);
    tc::bulk_load(sg.dK, &a.dw[fo], CH * LDF * 4, &sg.bar_ld);
    tc::bulk_load(sg.dG, &a.ddelta[fo], CH * LDF * 4, &sg.bar_ld);
    tc::mbar_arrive_expect_tx(&sg.bar_w, CH * LDF * 2);
    tc::bulk_load(sg.uh, &a.u[fo], CH * LDF * 2, &sg.bar_w);
  }
  __half* const wsh = reinterpret_cast<__half*>(s.At);
  static_assert(sizeof(s.At) == CH * LDF * sizeof(__half), "w takes the At tile's place");
  for (int e = tid; e < CH * DK / 8; e += NTH) {
    const int i = e >> 4, c8 = (e & 15) * 8;
    cp_async16(&wsh[i * LDF + c8], &a.w[w_off(chunk, h, a.HV) + i * DK + c8]);
  }
  // k, q, the gate and beta (one commit group with w), waited for after X and
  // Y, which do not read them.
  const RowScalars rows = load_chunk_issue<VEC, BetaT>(s, a.q, a.k, a.g, reinterpret_cast<const BetaT*>(a.beta),
                                                       cd.tok0, cd.len, hq, h, a.Hqk, a.HV);
  __syncthreads();  // the barrier set-up is visible
  if (!__syncthreads_and(tc::mbar_wait(&sg.bar_ld, 0))) {
    cp_async_wait<0>();
    if (tid == 0) {  // a wait ran out: record it and let the copies finish
      atomicExch(a.err, 7);
      tc::mbar_wait(&sg.bar_ld, 0);
      tc::mbar_wait(&sg.bar_w, 0);
    }
    return;
  }
  // Gate of (i, c) and (i, c + 1).
  auto gl2 = [&](int i, int c) -> float2 { return VEC ? s.g2(i, c) : make_float2(s.gs[i], s.gs[i]); };

  // v of this thread's accumulator positions, fetched now so that its latency
  // hides behind X, Y and dA.
  __nv_bfloat162 vpre[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = i0 + g + 8 * hr;
      vpre[nt][hr] = i < cd.len ? *reinterpret_cast<const __nv_bfloat162*>(
                                      &a.v[((size_t)(cd.tok0 + i) * a.HV + h) * DK + c0 + nt * 8 + 2 * t])
                                : __floats2bfloat162_rn(0.f, 0.f);
    }
  // X = T^T dw, Y = T^T dDelta (rows of block I, this warp's channels)
  float X[NT][4], Y[NT][4];
  zero_acc(X);
  zero_acc(Y);
  {
    const float* dw = sg.dK;
    const float* dd = sg.dG;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      if (kk < 2 * I) continue;
      const int ja = kk * 8 + t, jb = ja + 4;
      uint32_t av[4] = {tf32(s.T[ja * LDS + i0 + g]), tf32(s.T[ja * LDS + i0 + g + 8]),
                        tf32(s.T[jb * LDS + i0 + g]), tf32(s.T[jb * LDS + i0 + g + 8])};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int c = c0 + nt * 8 + g;
        uint32_t bx[2] = {tf32(dw[ja * LDF + c]), tf32(dw[jb * LDF + c])};
        uint32_t by[2] = {tf32(dd[ja * LDF + c]), tf32(dd[jb * LDF + c])};
        mma8(X[nt], av, bx);
        mma8(Y[nt], av, by);
      }
    }
  }
  __syncthreads();
  // The forward's At and dAqk (masked [64][64] FP32 tiles) into the dw staging
  // tile, which X and Y no longer read; they land during dA.
  float* const At = sg.dK;
  float* const dAqk = sg.dK + CH * LDS;
  if (tid == 0) {
    tc::mbar_arrive_expect_tx(&sg.bar_u, 2 * CH * LDS * 4);
    tc::bulk_load(At, &a.amat[so], CH * LDS * 4, &sg.bar_u);
    tc::bulk_load(dAqk, &a.daqk[so], CH * LDS * 4, &sg.bar_u);
  }
  load_chunk_finish<VEC>(s, rows);  // (also makes w visible)
  // Partial dA over this warp's channels: X w^T + Y u^T.  (A thread whose
  // wait for u runs out computes on whatever the tile holds; the barrier
  // after dA turns that into an error return.)
  const bool u_ok = tc::mbar_wait(&sg.bar_w, 0);
  float dAacc[8][4];
  zero_acc(dAacc);
  {
    const __half* u = reinterpret_cast<const __half*>(sg.uh);
#pragma unroll
    for (int kk = 0; kk < NT; ++kk) {
      uint32_t ax[4] = {tf32(X[kk][0]), tf32(X[kk][2]), tf32(X[kk][1]), tf32(X[kk][3])};
      uint32_t ay[4] = {tf32(Y[kk][0]), tf32(Y[kk][2]), tf32(Y[kk][1]), tf32(Y[kk][3])};
      const int cc = c0 + kk * 8 + 2 * t;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        if (nt < 2 * I + 2) {
          const int j = nt * 8 + g;
          const float2 wv = __half22float2(*reinterpret_cast<const __half2*>(&wsh[j * LDF + cc]));
          const float2 uv = __half22float2(*reinterpret_cast<const __half2*>(&u[j * LDF + cc]));
          uint32_t bw[2] = {__float_as_uint(wv.x), __float_as_uint(wv.y)};
          uint32_t bu[2] = {__float_as_uint(uv.x), __float_as_uint(uv.y)};
          mma8(dAacc[nt], ax, bw);
          mma8(dAacc[nt], ay, bu);
        }
      }
    }
  }
  // dA = -strict_tril(sum over the four quarters) into s.T (T is no longer
  // read), in quarter order.  The last pass also forms sum_j dA_ij At_ij of its
  // rows (part of dbeta).
  float* sDA = s.T;
  if (qc == 0)
    acc_foreach(dAacc, [&](int r, int col, float& x) { sDA[(i0 + r) * LDS + col] = col < i0 + r ? -x : 0.f; });
  if (!__syncthreads_and(tc::mbar_wait(&sg.bar_u, 0) && u_ok)) {  // (At and dAqk have landed)
    if (tid == 0) {
      atomicExch(a.err, 7);
      tc::mbar_wait(&sg.bar_w, 0);
      tc::mbar_wait(&sg.bar_u, 0);
    }
    return;
  }
#pragma unroll
  for (int pass = 1; pass < 3; ++pass) {
    if (qc == pass)
      acc_foreach(dAacc, [&](int r, int col, float& x) {
        if (col < i0 + r) sDA[(i0 + r) * LDS + col] -= x;
      });
    __syncthreads();
  }
  if (qc == 3) {
    float p0 = 0.f, p1 = 0.f;
    acc_foreach(dAacc, [&](int r, int col, float& x) {
      const int i = i0 + r;
      if (col < i) {
        const float d = sDA[i * LDS + col] - x;
        sDA[i * LDS + col] = d;
        if (r < 8) p0 += d * At[i * LDS + col]; else p1 += d * At[i * LDS + col];
      }
    });
    p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
    p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
    p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
    p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
    if (t == 0) {
      sg.dbeta[4][i0 + g] = p0;
      sg.dbeta[4][i0 + g + 8] = p1;
    }
  }
  // dK, dG: this warp's rows and channels, accumulator layout.
  float dKr[NT][4], dGr[NT][4];
  // Row-local: dV, dbeta (X.Kp + Y.V), dKp' = beta X Gamma.
  {
    float db0 = 0.f, db1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = i0 + g + 8 * hr, c = c0 + nt * 8 + 2 * t;
        const float2 vv = __bfloat1622float2(vpre[nt][hr]);
        const float2 kv = s.k2(i, c), gv = gl2(i, c);
        const float bi = s.beta[i];
        const float x0 = X[nt][2 * hr], x1 = X[nt][2 * hr + 1];
        const float e0 = ex2(gv.x), e1 = ex2(gv.y);
        const float part = (x0 * kv.x * e0 + Y[nt][2 * hr] * vv.x) + (x1 * kv.y * e1 + Y[nt][2 * hr + 1] * vv.y);
        if (hr == 0) db0 += part; else db1 += part;
        const float dkp0 = bi * x0 * e0, dkp1 = bi * x1 * e1;
        dKr[nt][2 * hr] = dkp0;
        dKr[nt][2 * hr + 1] = dkp1;
        dGr[nt][2 * hr] = kv.x * dkp0;
        dGr[nt][2 * hr + 1] = kv.y * dkp1;
        if (i < cd.len)
          *reinterpret_cast<__nv_bfloat162*>(&a.dv[((size_t)(cd.tok0 + i) * a.HV + h) * DK + c]) =
              __floats2bfloat162_rn(bi * Y[nt][2 * hr], bi * Y[nt][2 * hr + 1]);
      }
    }
    db0 += __shfl_xor_sync(0xffffffffu, db0, 1);
    db0 += __shfl_xor_sync(0xffffffffu, db0, 2);
    db1 += __shfl_xor_sync(0xffffffffu, db1, 1);
    db1 += __shfl_xor_sync(0xffffffffu, db1, 2);
    if (t == 0) {
      sg.dbeta[qc][i0 + g] = db0;
      sg.dbeta[qc][i0 + g + 8] = db1;
    }
  }
  __syncthreads();  // dA complete
  if (!VEC) {
    // Scalar gate: both masked matrices are only read with the decay
    // exp(gc_i - gc_j) from here on, so it is applied once, in place.
    for (int e = tid; e < CH * CH; e += NTH) {
      const int i = e >> 6, j = e & (CH - 1);
      if (j <= i) {
        const float d = ex2(s.gs[i] - s.gs[j]);
        sDA[i * LDS + j] *= d;
        dAqk[i * LDS + j] *= d;
      }
    }
    __syncthreads();
  }
  auto kf = [&](int j, int c) { return s.k(j, c); };
  // dqs at this thread's accumulator positions, fetched ahead of the apply.
  float2 dqspre[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr)
      dqspre[nt][hr] = __ldg(reinterpret_cast<const float2*>(&a.dqs[toff + (i0 + g + 8 * hr) * DK + c0 + nt * 8 + 2 * t]));
  // dKp' += beta [dA (x) decay] K  and  dQ = dqs * Gamma + [dAqk (x) decay] K.
  {
    float Z0[NT][4], Z1[NT][4];
    zero_acc(Z0);
    zero_acc(Z1);
    left_apply2<VEC, NT>(s, sDA, dAqk, kf, Z0, Z1, I, c0);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = i0 + g + 8 * hr, c = c0 + nt * 8 + 2 * t;
        const float bi = s.beta[i];
        const float2 kv = s.k2(i, c), qv = s.q2(i, c), gv = gl2(i, c);
        const float v0 = bi * Z0[nt][2 * hr], v1 = bi * Z0[nt][2 * hr + 1];
        dKr[nt][2 * hr] += v0;
        dKr[nt][2 * hr + 1] += v1;
        dGr[nt][2 * hr] += kv.x * v0;
        dGr[nt][2 * hr + 1] += kv.y * v1;
        const float2 dqs = dqspre[nt][hr];
        const float dq0 = dqs.x * ex2(gv.x) + Z1[nt][2 * hr];
        const float dq1 = dqs.y * ex2(gv.y) + Z1[nt][2 * hr + 1];
        dGr[nt][2 * hr] += qv.x * dq0;
        dGr[nt][2 * hr + 1] += qv.y * dq1;
        if (a.dq_part) {
          *reinterpret_cast<float2*>(&a.dq_part[toff + i * DK + c]) = make_float2(dq0, dq1);
        } else if (i < cd.len) {
          *reinterpret_cast<__nv_bfloat162*>(&a.dq[((size_t)(cd.tok0 + i) * a.Hqk + hq) * DK + c]) =
              __floats2bfloat162_rn(dq0, dq1);
        }
      }
  }
  // dKd at this thread's accumulator positions, fetched ahead of the last apply.
  float2 dkdpre[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr)
      dkdpre[nt][hr] = __ldg(reinterpret_cast<const float2*>(&a.dkd[toff + (i0 + g + 8 * hr) * DK + c0 + nt * 8 + 2 * t]));
  // dKn' = [dAqk (x) decay]^T Q + [beta dA (x) decay]^T K.
  {
    float Z[NT][4];
    zero_acc(Z);
    right_apply2<VEC, NT>(s, dAqk, sDA, Z, I, c0);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = i0 + g + 8 * hr, c = c0 + nt * 8 + 2 * t;
        const float2 kv = s.k2(i, c);
        dKr[nt][2 * hr] += Z[nt][2 * hr];
        dKr[nt][2 * hr + 1] += Z[nt][2 * hr + 1];
        dGr[nt][2 * hr] -= kv.x * Z[nt][2 * hr];
        dGr[nt][2 * hr + 1] -= kv.y * Z[nt][2 * hr + 1];
      }
  }
  // gamma * dgamma of this thread's channel (the chunk-end term of dg), fetched
  // here so that its latency hides behind the dKd terms.
  float gdg = 0.f;
  if (VEC || tid < DK) {
    const int c = tid & (DK - 1);
    gdg = __ldg(&a.gam[((size_t)chunk * a.HV + h) * DK + c]) * __ldg(&a.dgam[((size_t)chunk * a.HV + h) * DK + c]);
  }
  // dKd terms, dk, and the column sums of Kd*dKd over this warp's rows.
  {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int c = c0 + nt * 8 + 2 * t;
      const float2 glast = gl2(CH - 1, c);
      float cs0 = 0.f, cs1 = 0.f;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = i0 + g + 8 * hr;
        const float2 kv = s.k2(i, c), gv = gl2(i, c), x = dkdpre[nt][hr];
        const float ed0 = ex2(glast.x - gv.x), ed1 = ex2(glast.y - gv.y);
        const float kd0 = kv.x * ed0, kd1 = kv.y * ed1;  // Kd = K * exp(gc_last - gc)
        const float dk0 = dKr[nt][2 * hr] + x.x * ed0, dk1 = dKr[nt][2 * hr + 1] + x.y * ed1;
        dGr[nt][2 * hr] -= kd0 * x.x;
        dGr[nt][2 * hr + 1] -= kd1 * x.y;
        cs0 += kd0 * x.x;
        cs1 += kd1 * x.y;
        if (a.dk_part) {
          *reinterpret_cast<float2*>(&a.dk_part[toff + i * DK + c]) = make_float2(dk0, dk1);
        } else if (i < cd.len) {
          *reinterpret_cast<__nv_bfloat162*>(&a.dk[((size_t)(cd.tok0 + i) * a.Hqk + hq) * DK + c]) =
              __floats2bfloat162_rn(dk0, dk1);
        }
      }
#pragma unroll
      for (int m = 4; m < 32; m <<= 1) {
        cs0 += __shfl_xor_sync(0xffffffffu, cs0, m);
        cs1 += __shfl_xor_sync(0xffffffffu, cs1, m);
      }
      if (g == 0) *reinterpret_cast<float2*>(&sg.col[I * DK + c]) = make_float2(cs0, cs1);
    }
  }
  // The gate adjoint dgc of this warp's positions into the (free) staging tile.
  float* dG = sg.dG;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr)
      *reinterpret_cast<float2*>(&dG[(i0 + g + 8 * hr) * LDF + c0 + nt * 8 + 2 * t]) =
          make_float2(dGr[nt][2 * hr], dGr[nt][2 * hr + 1]);
  __syncthreads();
  if (VEC) {
    // Reverse cumsum over rows: thread group r (128 threads, one channel each)
    // takes rows 16r .. 16r + 15, starting from the sums of the later groups.
    const int c = tid & (DK - 1), r = tid >> 7;
    float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 16; ++i) part[i & 3] += dG[(16 * r + i) * LDF + c];
    s.tmp[r * DK + c] = (part[0] + part[1]) + (part[2] + part[3]);
    __syncthreads();
    float acc = gdg + ((sg.col[c] + sg.col[DK + c]) + (sg.col[2 * DK + c] + sg.col[3 * DK + c]));
    for (int r2 = 3; r2 > r; --r2) acc += s.tmp[r2 * DK + c];
#pragma unroll
    for (int i = 16 * r + 15; i >= 16 * r; --i) {
      acc += dG[i * LDF + c];
      if (i < cd.len) a.dg[((size_t)(cd.tok0 + i) * a.HV + h) * DK + c] = acc;
    }
  } else {
    // Scalar gate: dg_i = sum_{i' >= i} rowsum(dgc)_i' + the chunk-end term
    // sum_c (gamma dgamma + colsum(Kd dKd)).  Row sums: four threads per row
    // (channels q4, q4 + 4, ...); the chunk-end term: one channel per thread,
    // reduced per warp.
    if (tid < 4 * CH) {
      const int row = tid >> 2, q4 = tid & 3;
      float acc = 0.f;
#pragma unroll 8
      for (int k = 0; k < DK / 4; ++k) acc += dG[row * LDF + q4 + 4 * k];
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (q4 == 0) sg.rowsum[row] = acc;
    }
    if (tid < DK) {
      const int c = tid;
      float e = gdg +
                ((sg.col[c] + sg.col[DK + c]) + (sg.col[2 * DK + c] + sg.col[3 * DK + c]));
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) e += __shfl_xor_sync(0xffffffffu, e, m);
      if (lane == 0) s.tmp[warp] = e;
    }
    __syncthreads();
    if (tid < 32) {
      // dg_i = e + sum_{i' >= i} rowsum_i': lane l holds rows 2l and 2l + 1,
      // the sums of the later lanes by a reverse shuffle scan (fixed order).
      const float e = (s.tmp[0] + s.tmp[1]) + (s.tmp[2] + s.tmp[3]);
      const float t1 = sg.rowsum[2 * tid + 1], t0 = sg.rowsum[2 * tid] + t1;
      float x = t0;  // becomes the sum of lanes tid .. 31
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, x, d);
        if (tid + d < 32) x += y;
      }
      float later = __shfl_down_sync(0xffffffffu, x, 1);  // lanes tid + 1 .. 31
      if (tid == 31) later = 0.f;
      const float base = e + later;
      if (2 * tid < cd.len) a.dg[(size_t)(cd.tok0 + 2 * tid) * a.HV + h] = base + t0;
      if (2 * tid + 1 < cd.len) a.dg[(size_t)(cd.tok0 + 2 * tid + 1) * a.HV + h] = base + t1;
    }
  }
  if (tid < cd.len)
    reinterpret_cast<BetaT*>(a.dbeta)[(size_t)(cd.tok0 + tid) * a.HV + h] =
        from_f<BetaT>(((sg.dbeta[0][tid] + sg.dbeta[1][tid]) + (sg.dbeta[2][tid] + sg.dbeta[3][tid])) + sg.dbeta[4][tid]);
}

// dq / dk of a Q/K head = FP32 sum over its value heads, rounded once.  With
// the in-kernel q/k L2 normalization the sums are the gradients dn of the
// normalized vectors n = x r (r = (sum x^2 + eps)^(-1/2), saved by the
// forward's pre-pass), and the raw gradient is dx = r (dn - n (n . dn)).
// One warp per token row (lane: channels 4 lane .. 4 lane + 3; the dot
// products summed by shuffles in a fixed order).
__global__ void __launch_bounds__(256) k_group_reduce(GroupReduceArgs a) {
  const int chunk = a.chunk_base + blockIdx.x, hq = blockIdx.y;
  const ChunkDesc cd = a.chunks[chunk];
  const int G = a.HV / a.Hqk;
  const int warp = threadIdx.x >> 5, lane = lane_id(), c = 4 * lane;
  for (int i = warp; i < cd.len; i += 8) {
    float4 sq = make_float4(0.f, 0.f, 0.f, 0.f), sk = sq;
    for (int gi = 0; gi < G; ++gi) {
      const size_t off = tile_off(chunk, hq * G + gi, a.HV) + (size_t)i * DK + c;
      const float4 x = *reinterpret_cast<const float4*>(a.dq_part + off);
      const float4 y = *reinterpret_cast<const float4*>(a.dk_part + off);
      sq.x += x.x, sq.y += x.y, sq.z += x.z, sq.w += x.w;
      sk.x += y.x, sk.y += y.y, sk.z += y.z, sk.w += y.w;
    }
    const size_t row = (size_t)(cd.tok0 + i) * a.Hqk + hq, o = row * DK + c;
    if (a.rq) {  // through the normalization's Jacobian
      auto jac = [&](float4& d, const __nv_bfloat16* x, float r) {
        const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + o));
        const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + o + 2));
        const float n0 = x01.x * r, n1 = x01.y * r, n2 = x23.x * r, n3 = x23.y * r;
        float dot = (n0 * d.x + n1 * d.y) + (n2 * d.z + n3 * d.w);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
        d = make_float4(r * (d.x - n0 * dot), r * (d.y - n1 * dot), r * (d.z - n2 * dot), r * (d.w - n3 * dot));
      };
      jac(sq, a.q, a.rq[row]);
      jac(sk, a.k, a.rk[row]);
    }
    *reinterpret_cast<__nv_bfloat162*>(a.dq + o) = __floats2bfloat162_rn(sq.x, sq.y);
    *reinterpret_cast<__nv_bfloat162*>(a.dq + o + 2) = __floats2bfloat162_rn(sq.z, sq.w);
    *reinterpret_cast<__nv_bfloat162*>(a.dk + o) = __floats2bfloat162_rn(sk.x, sk.y);
    *reinterpret_cast<__nv_bfloat162*>(a.dk + o + 2) = __floats2bfloat162_rn(sk.z, sk.w);
  }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
cudaError_t launch_grad_state(const GradStateArgs& a, int nchunks, cudaStream_t st) {
  if (nchunks == 0) return cudaSuccess;
  const size_t sm = sizeof(GradStateSmem) + 1024;
  cudaFuncSetAttribute(k_grad_state, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  k_grad_state<<<dim3(nchunks, a.HV), 256, sm, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_grad(const GradArgs& a, int nchunks, bool vec, bool beta_bf16, cudaStream_t st) {
  if (nchunks == 0) return cudaSuccess;
  const size_t sm = sizeof(GradSmem);
  dim3 grid(nchunks, a.HV);
  if (vec && beta_bf16) {
    cudaFuncSetAttribute(k_grad<true, __nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_grad<true, __nv_bfloat16><<<grid, GRAD_WARPS * 32, sm, st>>>(a);
  } else if (vec) {
    cudaFuncSetAttribute(k_grad<true, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_grad<true, float><<<grid, GRAD_WARPS * 32, sm, st>>>(a);
  } else if (beta_bf16) {
    cudaFuncSetAttribute(k_grad<false, __nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_grad<false, __nv_bfloat16><<<grid, GRAD_WARPS * 32, sm, st>>>(a);
  } else {
    cudaFuncSetAttribute(k_grad<false, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_grad<false, float><<<grid, GRAD_WARPS * 32, sm, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_group_reduce(const GroupReduceArgs& a, int nchunks, cudaStream_t st) {
  if (nchunks == 0) return cudaSuccess;
  k_group_reduce<<<dim3(nchunks, a.Hqk), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdr
