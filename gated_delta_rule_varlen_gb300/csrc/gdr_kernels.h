// gdr_kernels.h -- kernel argument blocks and launchers (internal to the library).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gdr {

struct ChunkDesc;
struct DocDesc;
struct SegDesc;

// Chunk-major intermediates: tiles [NC][HV][64][128] FP32, Aqk [NC][HV][64][64],
// Kd stored transposed per chunk ([NC][HV][128 c][64 j]), gamma [NC][HV][128],
// BF16 state tapes [NC][HV][128 x 128], chunk-major: element (v, c) of a tile at
// ((c / 8) * 128 + v) * 8 + c % 8 (S0 of each chunk; dS, the adjoint of its end state).
struct PrepArgs {
  const __nv_bfloat16 *q, *k, *v;
  const float* g;
  const void* beta;  // bf16 (KDA) or fp32 (GDN)
  const ChunkDesc* chunks;
  int Hqk, HV;
  __half *w, *qp, *kd, *aqk;  // FP16, dense rows (gdr_common.cuh)
  __half* u;                  // FP16, rows LDF apart
  float* gam;
  float *amat, *tmat;  // At and T per chunk ([64][64] FP32), or null when nothing is saved
  // In-kernel q/k L2 normalization (else null): the scales r [T][Hqk] of q and
  // k's rows; q and k are then the raw inputs and every product takes the
  // normalized rows (the scales applied in FP32).
  const float *rq, *rk;
  int chunk_base;      // block x works on chunk chunk_base + x
};

// The tensor-core prep of grouped GDN (one CTA per (chunk, Q/K head), all
// value heads of the group): the prep's arguments plus 3-D BF16 tensor maps
// of q, k ([T][Hqk][128]) and v ([T][HV][128]), boxes of 64 channels x 1 head
// x 64 tokens, 128-byte swizzle.
struct PrepTcArgs {
  PrepArgs p;
  CUtensorMap q_map, k_map, v_map;
  int* err;  // device error word (bounded waits)
};

struct WalkArgs {
  // 2-D FP16 tensor maps (rows x columns), 128-byte swizzle, boxes of 64 columns:
  CUtensorMap w_map;    // w        [NC*HV*64][128] FP16, 64 x 64 boxes
  CUtensorMap kdt_map;  // Kd^T     [NC*HV*128][64] FP16, 64 x 128 boxes
  CUtensorMap u_map;    // u        [NC*HV*64][128] FP16, pitch LDF, 64 x 64 boxes
  CUtensorMap qp_map;   // Q Gamma  [NC*HV*64][128] FP16, 64 x 64 boxes
  CUtensorMap aqk_map;  // Aqk      [NC*HV*64][64]  FP16, 64 x 64 boxes
  const SegDesc* segs;  // walk segments, the longest document's first
  int HV;
  const float* gam;
  const float* h0;   // [N][HV][128][128] or null
  __nv_bfloat16* tape;  // S0 per chunk (BF16, chunk-major), or null
  float* delta;      // Delta per chunk, or null
  float* ht;         // [N][HV][128][128] or null
  __nv_bfloat16* out;  // [T][HV][128]
  // Per-segment states [NSEG][HV][128][128] (S[c][v]) of split documents:
  float* smap;       // the segment's state map M (end state = M start + bias)
  float* sstart;     // the segment's start state
  float* sbias;      // the segment's end state from a zero start
  float scale;
  int* err;          // device error word
  int seg_base;      // segments seg_base + blockIdx.x / HV
  int mode;          // 0 the full walks, 1 the summary walks (blockIdx.y: role)
  // Full walks: the chunk range [m0, m1) of every segment (m0 even; m1 past
  // the end for all of it), and per (segment, head) the carry state
  // [NSEG][HV][128][128] that passes between the slices of a pipelined walk.
  int m0, m1;
  float* carry;
};


struct WalkBwdArgs {
  // The saved FP16 tiles as the forward walk reads them (64-column boxes, 128-byte swizzle):
  CUtensorMap w_map, kdt_map, qp_map, aqk_map;
  const SegDesc* segs;
  int HV;
  float scale;
  const float* gam;
  const __nv_bfloat16* dout;  // [T][HV][128]
  const float* dht;           // [N][HV][128][128] or null
  __nv_bfloat16* dstape;      // dS (adjoint of each chunk's end state), BF16
  float* ddelta;              // dDelta per chunk
  float* dh0;                 // or null
  float* dsend;               // per segment: the adjoint of its end state
  float* dsbias;              // per segment: its start adjoint from a zero end adjoint
  int* err;                   // device error word
  int seg_base;
  int mode;                   // 0 the full walks, 1 the summary walks (blockIdx.y: role)
  int m0, m1;                 // full walks: the chunk range, as for the forward walk
  float* carry;               // the carry adjoint between slices [NSEG][HV][128][128]
};

// Merges of the segment states of split documents (one CTA per (segment,
// head, 16-column slice); only a document's first segment works).
struct MergeArgs {
  const SegDesc* segs;
  int HV, seg_base;
  const float* smap;
  float* state;       // forward: start states; backward: end adjoints
  const float* bias;  // forward: end states from zero; backward: start adjoints from zero
};

struct GradStateArgs {
  const ChunkDesc* chunks;
  int HV;
  float scale;
  const __nv_bfloat16* dout;
  const __nv_bfloat16 *tape, *dstape;
  const float *delta, *ddelta;
  float *dqs, *dw, *dkd, *dgam;  // scratch outputs
  float* daqk;                   // scale * tril(dO Delta^T), [NC][HV][64][64]
  int* err;                      // device error word
  int chunk_base;                // block x works on chunk chunk_base + x
};

struct GradArgs {
  const __nv_bfloat16 *q, *k, *v;
  const float* g;
  const void* beta;
  const __nv_bfloat16* dout;
  const ChunkDesc* chunks;
  int Hqk, HV;
  float scale;
  const __half* w;  // FP16 [64][128] per chunk
  const __half* u;  // FP16 [64][LDF] per chunk
  const float *gam, *delta, *ddelta;
  const float *dqs, *dw, *dkd, *dgam, *daqk;
  const float *amat, *tmat;  // At and T of each chunk, saved by the forward
  // outputs
  __nv_bfloat16 *dq, *dk, *dv;   // dq/dk written directly when HV == Hqk
  float *dq_part, *dk_part;      // [NC][HV][64][128] per value head when HV > Hqk
  float* dg;
  void* dbeta;
  int* err;  // device error word
  int chunk_base;  // block x works on chunk chunk_base + x
};

struct GroupReduceArgs {
  const ChunkDesc* chunks;
  int Hqk, HV;
  const float *dq_part, *dk_part;
  __nv_bfloat16 *dq, *dk;
  // In-kernel q/k L2 normalization (else null): the raw q, k and the scales r
  // [T][Hqk] of their normalized copies.
  const __nv_bfloat16 *q, *k;
  const float *rq, *rk;
  int chunk_base;  // block x works on chunk chunk_base + x
};

// In-kernel q/k L2 normalization (forward pre-pass): each (token, Q/K head)
// vector x of q and k -> n = x r (BF16), r = (sum x^2 + eps)^(-1/2) (FP32).
struct L2NormArgs {
  const __nv_bfloat16 *q, *k;
  __nv_bfloat16 *qn, *kn;
  float *rq, *rk;
  int64_t rows;  // T * Hqk
};

cudaError_t launch_prep(const PrepArgs& a, int nchunks, cudaStream_t st);  // KDA (per-channel gate)
cudaError_t launch_prep_gdn(const PrepTcArgs& a, int nchunks, cudaStream_t st);
cudaError_t launch_walk_fwd_v(const WalkArgs& a, int nsegs, cudaStream_t st);
cudaError_t launch_merge(const MergeArgs& a, int nsegs, bool backward, cudaStream_t st);
cudaError_t launch_walk_bwd_v(const WalkBwdArgs& a, int nsegs, cudaStream_t st);
cudaError_t launch_grad_state(const GradStateArgs& a, int nchunks, cudaStream_t st);
cudaError_t launch_grad(const GradArgs& a, int nchunks, bool vec, bool beta_bf16, cudaStream_t st);
cudaError_t launch_group_reduce(const GroupReduceArgs& a, int nchunks, cudaStream_t st);
cudaError_t launch_l2norm(const L2NormArgs& a, cudaStream_t st);

}  // namespace gdr
