// gdr_api.cu -- the C ABI (include/gdr.h): validation, planning, workspace
// layout, the saved-buffer stamp, and the launch sequences.
#include <algorithm>
#include <climits>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <string>
#include <map>
#include <vector>
#include <cstdio>

#include <cudaTypedefs.h>

#include "../../include/gdr.h"
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "gdr_tc.cuh"

namespace gdr {
namespace {

constexpr size_t kAlign = 256;
constexpr int kRankLimit = 4096;  // documents ranked longest-first on the device up to this count

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// ---------------------------------------------------------------------------
// Header at the start of a saved buffer: which saving forward filled it.  The
// saving forward's planning kernel writes it; the backward compares it on the
// device with what its own arguments imply (kStaleCode in the device error
// word on a mismatch).  The buffer's contents are position-independent, so a
// saved buffer copied to another address stays valid.
struct SavedHeader {
  uint64_t magic;
  int64_t T;
  int32_t N, Hqk, HV, variant, lseg, l2;
  uint64_t cu_hash;
  uint64_t counter;  // which saving forward of this process wrote it (1, 2, ...)
};
constexpr uint64_t kSavedMagic = 0x3145564153524447ull;
constexpr int kStaleCode = 8;

// Planning kernel: document and chunk tables from the device cu_seqlens, and
// the longest-first document order for the walks (the LPT rule of PR #7723
// "perf(cake_gdn): prefetch offset adjoint walk, default LPT segment plan",
// applied here to whole documents on one GPU).  Chunks are numbered in that
// order (the longest document's chunks first), so that any run of documents
// in it owns one contiguous range of chunks.  Ties go to the lower document
// index; above kRankLimit documents the order is the given one.  One block; no
// host copy.  plan_ranks() on the host reproduces the same order.  A saving
// forward also writes the saved buffer's header (hdr_out).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_plan(const int* __restrict__ cu, int N, int lseg, DocDesc* docs,
                                               ChunkDesc* chunks, int* order, SegDesc* segs, SavedHeader hdr,
                                               SavedHeader* hdr_out) {
  __shared__ int part[1024], spart[1024];
  if (hdr_out && threadIdx.x == 0) *hdr_out = hdr;
  __shared__ int lens[kRankLimit];
  __shared__ int ord[kRankLimit];
  const int tid = threadIdx.x, nt = blockDim.x;
  const bool ranked = N <= kRankLimit;
  if (ranked) {
    for (int n = tid; n < N; n += nt) lens[n] = cu[n + 1] - cu[n];
    __syncthreads();
    for (int n = tid; n < N; n += nt) {
      const int ln = lens[n];
      int rank = 0;
      for (int m = 0; m < N; ++m) rank += (lens[m] > ln) || (lens[m] == ln && m < n);
      ord[rank] = n;
      order[rank] = n;
    }
  } else {
    for (int n = tid; n < N; n += nt) order[n] = n;
  }
  __syncthreads();
  auto doc_at = [&](int r) { return ranked ? ord[r] : r; };
  // Chunk and segment offsets: prefix sums of chunk and segment counts over the ranks.
  const int per = (N + nt - 1) / nt;
  const int r0 = min(N, tid * per), r1 = min(N, r0 + per);
  int sum = 0, ssum = 0;
  for (int r = r0; r < r1; ++r) {
    const int n = doc_at(r);
    const int nch = (cu[n + 1] - cu[n] + CH - 1) / CH;
    sum += nch;
    ssum += nch == 0 ? 1 : (nch + lseg - 1) / lseg;
  }
  part[tid] = sum;
  spart[tid] = ssum;
  __syncthreads();
  if (tid == 0) {
    int acc = 0, sacc = 0;
    for (int i = 0; i < nt; ++i) {
      const int v = part[i], sv = spart[i];
      part[i] = acc;
      spart[i] = sacc;
      acc += v;
      sacc += sv;
    }
  }
  __syncthreads();
  int c = part[tid], sg = spart[tid];
  for (int r = r0; r < r1; ++r) {
    const int n = doc_at(r);
    const int tok0 = cu[n], len = cu[n + 1] - tok0, nch = (len + CH - 1) / CH;
    docs[n] = DocDesc{tok0, len, c, nch};
    for (int j = 0; j < nch; ++j) chunks[c + j] = ChunkDesc{tok0 + CH * j, min(CH, len - CH * j), n, j};
    const int nseg = nch == 0 ? 1 : (nch + lseg - 1) / lseg;
    const int base = nseg > 0 ? nch / nseg : 0, rem = nseg > 0 ? nch % nseg : 0;
    for (int i = 0; i < nseg; ++i) {
      const int off = i * base + min(i, rem), cnt = base + (i < rem ? 1 : 0);
      const int t0 = tok0 + CH * off;
      segs[sg + i] = SegDesc{n, t0, min(CH * cnt, len - CH * off), c + off, cnt, i, nseg, sg};
    }
    c += nch;
    sg += nseg;
  }
}

// The backward's check of a saved buffer's header (one thread): a mismatch
// with the expected header (the counter only when `with_counter`) sets
// kStaleCode in the device error word.
__global__ void k_check_header(SavedHeader want, const SavedHeader* __restrict__ have, int with_counter, int* err) {
  if (threadIdx.x != 0) return;
  const SavedHeader h = *have;
  const bool ok = h.magic == want.magic && h.T == want.T && h.N == want.N && h.Hqk == want.Hqk && h.HV == want.HV &&
                  h.variant == want.variant && h.lseg == want.lseg && h.l2 == want.l2 && h.cu_hash == want.cu_hash &&
                  (!with_counter || h.counter == want.counter);
  if (!ok) atomicExch(err, kStaleCode);
}

// Host copy of the plan's document order, and the split of the backward into
// document groups that run on streams of their own: each of the first
// kMaxSolo documents (longest first) with at least kSoloChunks chunks is a
// group, and the remaining documents form one more.  A group's chunks are one
// contiguous range (k_plan numbers them in this order).
constexpr int kMaxGroups = 4;
constexpr int kMaxSolo = kMaxGroups - 1;
constexpr int kSoloChunks = 64;
struct DocGroup {
  int r0, r1;        // ranks [r0, r1) of order[]
  int64_t c0, c1;    // chunks [c0, c1)
  int64_t tokens;
  int64_t s0 = 0, s1 = 0;  // segments [s0, s1) (k_plan numbers them in rank order)
  bool split = false;       // some document of the group has more than one segment
};
std::vector<DocGroup> plan_groups(int32_t N, const int32_t* cu) {
  std::vector<int> ord(N);
  for (int n = 0; n < N; ++n) ord[n] = n;
  if (N <= kRankLimit)
    std::stable_sort(ord.begin(), ord.end(), [&](int x, int y) { return cu[x + 1] - cu[x] > cu[y + 1] - cu[y]; });
  std::vector<DocGroup> gr;
  int64_t c = 0;
  int r = 0;
  while (r < N) {
    const int n = ord[r];
    const int64_t nch = (cu[n + 1] - cu[n] + CH - 1) / CH;
    if ((int)gr.size() < kMaxSolo && nch >= kSoloChunks) {
      gr.push_back(DocGroup{r, r + 1, c, c + nch, (int64_t)(cu[n + 1] - cu[n])});
      c += nch;
      ++r;
      continue;
    }
    DocGroup g{r, N, c, c, 0};
    for (; r < N; ++r) {
      const int m = ord[r];
      g.c1 += (cu[m + 1] - cu[m] + CH - 1) / CH;
      g.tokens += cu[m + 1] - cu[m];
    }
    gr.push_back(g);
  }
  if (gr.size() <= 1) {
    int64_t nc = 0, tok = 0;
    for (int n = 0; n < N; ++n) {
      nc += (cu[n + 1] - cu[n] + CH - 1) / CH;
      tok += cu[n + 1] - cu[n];
    }
    return {DocGroup{0, N, 0, nc, tok}};
  }
  return gr;
}

// Segments of the state walks.  A chain (document, value head) is walked one
// chunk after another; a long document is split into segments of about
// `lseg` chunks whose walks run in parallel: summary walks give each
// segment's affine map of its start state, a merge chains the start states,
// and the full walks of all segments then run from their start states (the
// segment plan of PR #7723, "perf(cake_gdn): prefetch offset adjoint walk,
// default LPT segment plan", on one GPU).  Splitting adds walk work (the
// summary walks), so it pays only when the longest document's chain, walked
// whole, outlasts the work of all the other documents spread over the SMs
// (which the document groups run beside it): per chunk, the forward and
// backward walk steps take about kWalkStepNs on the chain, and a chunk of one
// head costs about kChunkHeadNs of SM time over the whole step (prep, walks,
// gradients), both measured on GB300.  A longest document that would walk
// pipelined (a group of its own, longer than a slice) overlaps its walk with
// its own prep and gradient work too, so that work counts on the other side.
// A split pack gets segments of lseg = max(kMinSegChunks, chunks x heads /
// SMs), which about fill the SMs.
constexpr int kMinSegChunks = 64;
constexpr int kNoSplit = 1 << 30;
constexpr double kWalkStepNs = 7700.0, kChunkHeadNs = 50000.0;
std::atomic<int> g_seg_chunks{0};  // gdr_set_segment_chunks: 0 = choose

int sm_count();
int slice_chunks();

int segment_chunks(int32_t N, const int32_t* cu, int32_t HV) {
  const int forced = g_seg_chunks.load();
  if (forced > 0) return forced;
  int64_t total = 0, longest = 0;
  for (int32_t n = 0; n < N; ++n) {
    const int64_t nch = (cu[n + 1] - cu[n] + CH - 1) / CH;
    total += nch;
    longest = std::max(longest, nch);
  }
  const int64_t sms = sm_count();
  const double chain_ns = (double)longest * kWalkStepNs;
  const bool own = longest >= kSoloChunks && longest > slice_chunks();
  const double others_ns = (double)(own ? total : total - longest) * HV * kChunkHeadNs / (double)sms;
  if (chain_ns <= others_ns) return kNoSplit;
  const int64_t l = std::max<int64_t>(kMinSegChunks, (total * HV + sms - 1) / sms);
  return longest <= l ? kNoSplit : (int)l;
}

int64_t doc_segments(int64_t nch, int lseg) { return nch == 0 ? 1 : (nch + lseg - 1) / lseg; }

// Segment ranges of the groups (the documents' segments in rank order) and
// the total segment count.
int64_t assign_segments(std::vector<DocGroup>& groups, int32_t N, const int32_t* cu, int lseg) {
  std::vector<int> ord(N);
  for (int n = 0; n < N; ++n) ord[n] = n;
  if (N <= kRankLimit)
    std::stable_sort(ord.begin(), ord.end(), [&](int x, int y) { return cu[x + 1] - cu[x] > cu[y + 1] - cu[y]; });
  std::vector<int64_t> first(N + 1, 0);
  std::vector<bool> split(N, false);
  for (int r = 0; r < N; ++r) {
    const int64_t nch = (cu[ord[r] + 1] - cu[ord[r]] + CH - 1) / CH;
    const int64_t ns = doc_segments(nch, lseg);
    first[r + 1] = first[r] + ns;
    split[r] = ns > 1;
  }
  for (DocGroup& g : groups) {
    g.s0 = first[g.r0];
    g.s1 = first[g.r1];
    g.split = false;
    for (int r = g.r0; r < g.r1; ++r) g.split = g.split || split[r];
  }
  return first[N];
}

// ---------------------------------------------------------------------------
// Workspace layout.
// ---------------------------------------------------------------------------
struct Layout {
  int64_t NC = 0, NSEG = 0;
  size_t header = 0;                             // SavedHeader (saved buffers)
  size_t bdocs = 0, bchunks = 0, border = 0, bsegs = 0;  // the backward's own plan (scratch)
  size_t docs = 0, chunks = 0, order = 0, segs = 0, w = 0, u = 0, qp = 0, kd = 0, delta = 0, aqk = 0, amat = 0,
         tmat = 0, gam = 0, tape = 0, smap = 0, sstart = 0, sbias = 0, fcarry = 0, bcarry = 0;
  size_t saved_total = 0;
  size_t qn = 0, kn = 0, rq = 0, rk = 0;  // in-kernel q/k L2 normalization
  size_t dstape = 0, ddelta = 0, dqs = 0, dw = 0, dkd = 0, dgam = 0, daqk = 0, dqp = 0, dkp = 0, dsend = 0, dsbias = 0;
  size_t bwd_total = 0;
};

// NSEG: segments of the walks (equal to N when no document is split); the
// per-segment state buffers are only laid out when some document is.
Layout make_layout(int64_t T, int64_t NC, int32_t N, int32_t Hqk, int32_t HV, bool l2, int64_t NSEG) {
  const bool grouped = HV != Hqk || l2;  // FP32 dq / dk partials reduced (and normalized back) per Q/K head
  Layout L;
  L.NC = NC;
  L.NSEG = NSEG;
  const bool split = NSEG > N;
  const size_t segstate = split ? (size_t)NSEG * HV * DK * DK * sizeof(float) : 0;
  const size_t tile = (size_t)NC * HV * CH * DK * sizeof(float);
  const size_t vec = (size_t)NC * HV * DK * sizeof(float);
  const size_t st = (size_t)NC * HV * DK * DK * sizeof(uint16_t);  // BF16 state tapes
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.header = take(sizeof(SavedHeader));
  L.docs = take((size_t)std::max(N, 1) * sizeof(DocDesc));
  L.chunks = take((size_t)std::max<int64_t>(NC, 1) * sizeof(ChunkDesc));
  L.order = take((size_t)std::max(N, 1) * sizeof(int));
  L.segs = take((size_t)std::max<int64_t>(NSEG, 1) * sizeof(SegDesc));
  L.smap = take(segstate);    // each split segment's state map (the backward merge needs it too)
  L.sstart = take(segstate);  // start state of each segment
  L.sbias = take(segstate);   // each segment's end state from a zero start
  L.fcarry = take((size_t)std::max<int64_t>(NSEG, 1) * HV * DK * DK * sizeof(float));  // pipelined walks
  L.w = take((size_t)NC * HV * CH * DK * sizeof(__half));
  L.u = take((size_t)NC * HV * CH * LDF * sizeof(__half));
  L.qp = take((size_t)NC * HV * CH * DK * sizeof(__half));
  L.kd = take((size_t)NC * HV * DK * CH * sizeof(__half));
  L.delta = take(tile);
  L.aqk = take((size_t)NC * HV * CH * CH * sizeof(__half));
  L.amat = take((size_t)NC * HV * CH * LDS * sizeof(float));
  L.tmat = take((size_t)NC * HV * CH * LDS * sizeof(float));
  L.gam = take(vec);
  L.tape = take(st);
  if (l2) {
    L.qn = take((size_t)T * Hqk * DK * 2);
    L.kn = take((size_t)T * Hqk * DK * 2);
    L.rq = take((size_t)T * Hqk * 4);
    L.rk = take((size_t)T * Hqk * 4);
  }
  L.saved_total = o;
  o = 0;
  // The backward plans again into its scratch, so that no index it follows
  // comes from the saved buffer.
  L.bdocs = take((size_t)std::max(N, 1) * sizeof(DocDesc));
  L.bchunks = take((size_t)std::max<int64_t>(NC, 1) * sizeof(ChunkDesc));
  L.border = take((size_t)std::max(N, 1) * sizeof(int));
  L.bsegs = take((size_t)std::max<int64_t>(NSEG, 1) * sizeof(SegDesc));
  L.dstape = take(st);
  L.ddelta = take((size_t)NC * HV * CH * LDF * sizeof(float));
  L.dqs = take(tile);
  L.dw = take((size_t)NC * HV * CH * LDF * sizeof(float));
  L.dkd = take(tile);
  L.dgam = take(vec);
  L.daqk = take((size_t)NC * HV * CH * LDS * sizeof(float));
  L.dsend = take(segstate);   // adjoint of each segment's end state
  L.dsbias = take(segstate);  // each segment's start adjoint from a zero end adjoint
  L.bcarry = take((size_t)std::max<int64_t>(NSEG, 1) * HV * DK * DK * sizeof(float));  // pipelined walks
  if (grouped) {
    L.dqp = take(tile);
    L.dkp = take(tile);
  }
  L.bwd_total = o;
  return L;
}

// Validates cu_seqlens_host and counts chunks.
gdr_status plan_host(int64_t T, int32_t N, const int32_t* cu, int64_t* NC) {
  if (N < 0 || T < 0) return GDR_INVALID_ARG;
  if (!cu) return GDR_INVALID_ARG;
  if (cu[0] != 0 || (int64_t)cu[N] != T) return GDR_BAD_CU_SEQLENS;
  if (T > INT32_MAX) return GDR_INVALID_ARG;
  int64_t nc = 0;
  for (int32_t n = 0; n < N; ++n) {
    if (cu[n + 1] < cu[n]) return GDR_BAD_CU_SEQLENS;
    nc += (cu[n + 1] - cu[n] + CH - 1) / CH;
  }
  *NC = nc;
  return GDR_OK;
}

uint64_t hash_cu(const int32_t* cu, int32_t N) {
  uint64_t h = 1469598103934665603ull;
  for (int32_t i = 0; i <= N; ++i) {
    h ^= (uint32_t)cu[i];
    h *= 1099511628211ull;
  }
  return h;
}

// Host registry of the saved buffers this process filled, keyed by address:
// the stamp of the last saving forward into each.  The backward rejects,
// before enqueueing anything, a registered buffer whose stamp does not match
// its arguments; an unregistered one (copied to another address, or filled
// by another process) is left to the device-side header check alone.
struct Stamp {
  int64_t T;
  int32_t N, Hqk, HV, variant, lseg;
  bool l2;
  uint64_t cu_hash;
  uint64_t counter;
};
std::mutex g_stamp_mu;
std::unordered_map<const void*, Stamp> g_stamps;
std::atomic<uint64_t> g_save_counter{0};

enum class StampState { kUnknown, kMatch, kMismatch };

void stamp_set(const void* saved, const Stamp& s) {
  std::lock_guard<std::mutex> lk(g_stamp_mu);
  g_stamps[saved] = s;
}
// On kMatch, *counter is the registered forward's counter.
StampState stamp_check(const void* saved, const Stamp& s, uint64_t* counter) {
  std::lock_guard<std::mutex> lk(g_stamp_mu);
  auto it = g_stamps.find(saved);
  if (it == g_stamps.end()) return StampState::kUnknown;
  const Stamp& r = it->second;
  const bool same = r.T == s.T && r.N == s.N && r.Hqk == s.Hqk && r.HV == s.HV && r.variant == s.variant &&
                    r.lseg == s.lseg && r.l2 == s.l2 && r.cu_hash == s.cu_hash;
  if (!same) return StampState::kMismatch;
  *counter = r.counter;
  return StampState::kMatch;
}

SavedHeader header_of(const Stamp& s) {
  SavedHeader h{};
  h.magic = kSavedMagic;
  h.T = s.T;
  h.N = s.N;
  h.Hqk = s.Hqk;
  h.HV = s.HV;
  h.variant = s.variant;
  h.lseg = s.lseg;
  h.l2 = s.l2 ? 1 : 0;
  h.cu_hash = s.cu_hash;
  h.counter = s.counter;
  return h;
}

gdr_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDR_CUDA_ERROR;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return GDR_CUDA_ERROR;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return GDR_CUDA_ERROR;
  if (major != 10 || minor != 3) return GDR_UNSUPPORTED;
  return GDR_OK;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 152;
}

bool aligned(const void* p) { return ((uintptr_t)p % kAlign) == 0; }
// Tensors the kernels copy in 16-byte pieces (q, k, v, g, dout) or store in
// pairs must start on these boundaries.
bool aligned_to(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

gdr_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GDR_OK : GDR_CUDA_ERROR; }

// ---------------------------------------------------------------------------
// TMA tensor maps (encoded on the host; the driver entry point is fetched
// through the runtime, so the library does not link the driver library).
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// rows x cols FP16 tensor whose rows are `pitch` elements apart (default:
// dense); boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool fp16_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
              uint64_t pitch = 0) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {(pitch ? pitch : cols) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [T][H][128] BF16 tensor (q, k or v) read one head at a time: boxes of 64
// channels x 1 head x 64 tokens, 128-byte swizzle (zero fill past T).
bool bf16_head_map(CUtensorMap* map, const void* base, uint64_t T, uint64_t H) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {DK, H, T};
  cuuint64_t strides[2] = {DK * 2, H * DK * 2};
  cuuint32_t box[3] = {64, 1, CH};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Device error word: a kernel whose bounded wait runs out writes a non-zero
// code here (and skips the work that depended on the wait).
// One warp waits on a barrier that nothing completes, with the walks' bounded
// wait; when the limit runs out the timeout is recorded in the error word.
__global__ void k_selftest_wait(uint64_t limit_ns, int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, limit_ns)) atomicExch(err, 5);
}

static __device__ int g_device_error;
std::mutex g_err_mu;
int* g_err_ptr[64] = {};

int* device_error_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}


// ---------------------------------------------------------------------------
// Opt-in per-kernel timing for benchmarks: while enabled, every launch is
// bracketed by a pair of CUDA events recorded on the launch's stream.
// ---------------------------------------------------------------------------
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
  double units;  // token-heads the launch works on
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;

void prof_clear_locked() {
  for (auto& r : g_prof) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  g_prof.clear();
}

// Kernel launches enqueued by the compute calls since the library was loaded
// (every launch site opens a ProfScope).
std::atomic<uint64_t> g_launches{0};
// While set, every call runs all its launches on the caller's stream (its
// document groups one after another): per-kernel timing without overlap.
std::atomic<bool> g_serial{false};

struct ProfScope {
  cudaStream_t st;
  bool on;
  ProfScope(const char* name, cudaStream_t s, double units = 0) : st(s), on(false) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return;
    ProfRec r{name, nullptr, nullptr, units};
    if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return;
    cudaEventRecord(r.a, st);
    g_prof.push_back(r);
    on = true;
  }
  ~ProfScope() {
    if (!on) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    cudaEventRecord(g_prof.back().b, st);
  }
};

// ---------------------------------------------------------------------------
// Streams the backward's document groups run on (per device, created once,
// the first with the highest priority), and the fork from / join back to the
// caller's stream around them.  A single group runs on the caller's stream.
// ---------------------------------------------------------------------------
std::mutex g_lane_mu;
// Lane i is group i's first lane (its walks), lane kMaxGroups + i its second
// (the prep or the gradient kernels of a pipelined walk), at a lower priority
// so that the walk slices win the SMs that free up.
constexpr int kLanes = 2 * kMaxGroups;
cudaStream_t g_lanes[64][kLanes] = {};

const cudaStream_t* lanes_for_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_lane_mu);
  if (!g_lanes[dev][kLanes - 1]) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
    for (int i = 0; i < kLanes; ++i) {
      if (g_lanes[dev][i]) continue;
      const int prio = std::min(least, greatest + i);  // numerically lower = higher priority
      if (cudaStreamCreateWithPriority(&g_lanes[dev][i], cudaStreamNonBlocking, prio) != cudaSuccess) {
        g_lanes[dev][i] = nullptr;
        return nullptr;
      }
    }
  }
  return g_lanes[dev];
}

class Fork {
 public:
  // n groups; `second`: some group also uses its second lane.
  Fork(cudaStream_t main, int n, bool second = false)
      : main_(main), n_(g_serial.load() ? 1 : n), on_(!g_serial.load() && (n > 1 || second)) {}
  Fork(const Fork&) = delete;
  Fork& operator=(const Fork&) = delete;
  // Makes every lane wait for the work already on the caller's stream.
  bool begin() {
    if (!on_) return true;
    lanes_ = lanes_for_device();
    if (!lanes_) return false;
    cudaEvent_t ev;
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return false;
    bool ok = cudaEventRecord(ev, main_) == cudaSuccess;
    for (int i = 0; ok && i < n_; ++i)
      ok = cudaStreamWaitEvent(lanes_[i], ev, 0) == cudaSuccess &&
           cudaStreamWaitEvent(lanes_[kMaxGroups + i], ev, 0) == cudaSuccess;
    cudaEventDestroy(ev);
    forked_ = ok;
    return ok;
  }
  cudaStream_t lane(int i) const { return on_ ? lanes_[i] : main_; }
  cudaStream_t lane2(int i) const { return on_ ? lanes_[kMaxGroups + i] : main_; }
  // Makes `to` wait for the work enqueued so far on `from`.
  static bool link(cudaStream_t from, cudaStream_t to) {
    if (from == to) return true;
    cudaEvent_t ev;
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return false;
    const bool ok = cudaEventRecord(ev, from) == cudaSuccess && cudaStreamWaitEvent(to, ev, 0) == cudaSuccess;
    cudaEventDestroy(ev);
    return ok;
  }
  // Makes the caller's stream wait for everything enqueued on the lanes.
  bool join() {
    if (!forked_) return true;
    forked_ = false;
    bool ok = true;
    for (int i = 0; i < n_; ++i) ok = link(lanes_[i], main_) && link(lanes_[kMaxGroups + i], main_) && ok;
    return ok;
  }
  ~Fork() { join(); }

 private:
  cudaStream_t main_;
  int n_;
  bool on_;
  const cudaStream_t* lanes_ = nullptr;
  bool forked_ = false;
};

// Slices of a pipelined walk (chunks, even): the walk of a group that holds
// one unsplit document longer than a slice runs slice by slice (the state, or
// the adjoint, passed on exactly in FP32 through a carry buffer), so that the
// forward walk starts once the first slice is prepared, and the backward's
// gradient kernels of a slice run while the walk goes on with the next one.
constexpr int kSliceChunks = 128;
std::atomic<int> g_slice_chunks{0};  // gdr_set_slice_chunks: 0 = kSliceChunks
int slice_chunks() {
  const int v = g_slice_chunks.load();
  return v > 0 ? v : kSliceChunks;
}
bool pipelined(const DocGroup& G, int S) { return !G.split && G.r1 - G.r0 == 1 && G.c1 - G.c0 > S; }

// Slice boundaries of a pipelined walk over nch > S chunks: a first and a last
// slice of S / div chunks (the forward walk starts after less prep, the
// backward's gradient kernels after less walk, and the slice that runs alone
// at the end is short), the chunks between them in equal slices of about S;
// every slice starts at an even chunk.  A walk too short for that is cut into
// slices of S.  Measured on GB300: div = 2 for the forward, 4 for the
// backward (div = 8 slower for both).
std::vector<int> slice_bounds(int nch, int S, int div) {
  const int e = std::max(2, (S / div) & ~1);
  std::vector<int> b{0};
  if (nch < 2 * e + 2) {
    for (int m = S; m < nch; m += S) b.push_back(m);
    b.push_back(nch);
    return b;
  }
  const int last = (nch - e) & ~1;
  b.push_back(e);
  const int L = last - e, k = (L + S - 1) / S;
  for (int j = 1; j < k; ++j) b.push_back((e + (int)((int64_t)L * j / k)) & ~1);
  if (last > b.back()) b.push_back(last);
  b.push_back(nch);
  return b;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}
template <typename T>
const T* at(const void* base, size_t off) {
  return reinterpret_cast<const T*>(static_cast<const char*>(base) + off);
}

gdr_status workspace_bytes(int64_t T, int32_t Hqk, int32_t HV, int32_t N, const int32_t* cu, int l2,
                           size_t* saved_bytes, size_t* scratch_bytes) {
  if (Hqk <= 0 || HV <= 0 || HV % Hqk != 0) return GDR_INVALID_ARG;
  int64_t NC = 0;
  const gdr_status st = plan_host(T, N, cu, &NC);
  if (st != GDR_OK) return st;
  std::vector<DocGroup> groups = plan_groups(N, cu);
  const int64_t NSEG = assign_segments(groups, N, cu, segment_chunks(N, cu, HV));
  const Layout L = make_layout(T, NC, N, Hqk, HV, l2 != 0, NSEG);
  if (saved_bytes) *saved_bytes = L.saved_total;
  if (scratch_bytes) *scratch_bytes = L.bwd_total;
  return GDR_OK;
}

gdr_status fwd_impl(int variant, const void* q, const void* k, const void* v, const float* g, const void* beta,
                    const int32_t* cu, const int32_t* cu_host, int32_t N, int64_t T, int32_t Hqk, int32_t HV,
                    float scale, int l2, const float* h0, void* out, float* ht, void* saved, size_t saved_bytes,
                    int save_for_bwd, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  if (Hqk <= 0 || HV <= 0 || HV % Hqk != 0) return GDR_INVALID_ARG;
  int64_t NC = 0;
  gdr_status st = plan_host(T, N, cu_host, &NC);
  if (st != GDR_OK) return st;
  if (N == 0) return GDR_OK;
  if (!cu) return GDR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return GDR_INVALID_ARG;
  if (!aligned_to(q, 16) || !aligned_to(k, 16) || !aligned_to(v, 16) || !aligned_to(g, 16) || !aligned_to(out, 4))
    return GDR_INVALID_ARG;
  if (save_for_bwd && !saved) return GDR_INVALID_ARG;
  const int lseg = segment_chunks(N, cu_host, HV);
  std::vector<DocGroup> groups = plan_groups(N, cu_host);
  const int64_t NSEG = assign_segments(groups, N, cu_host, lseg);
  const Layout L = make_layout(T, NC, N, Hqk, HV, l2 != 0, NSEG);
  void* base = saved ? saved : scratch;
  const size_t have = saved ? saved_bytes : scratch_bytes;
  if (!base) return GDR_INVALID_ARG;
  if (!aligned(base)) return GDR_INVALID_ARG;
  if (have < L.saved_total) return GDR_WORKSPACE_TOO_SMALL;
  st = check_device();
  if (st != GDR_OK) return st;

  DocDesc* docs = at<DocDesc>(base, L.docs);
  ChunkDesc* chunks = at<ChunkDesc>(base, L.chunks);
  int* order = at<int>(base, L.order);
  SegDesc* segs = at<SegDesc>(base, L.segs);
  Stamp stamp{T, N, Hqk, HV, variant, lseg, l2 != 0, hash_cu(cu_host, N), 0};
  if (save_for_bwd) stamp.counter = g_save_counter.fetch_add(1) + 1;
  {
    ProfScope ps("plan", stream);
    k_plan<<<1, 1024, 0, stream>>>(cu, N, std::min(lseg, kNoSplit), docs, chunks, order, segs, header_of(stamp),
                                   save_for_bwd ? at<SavedHeader>(base, L.header) : nullptr);
  }
  if (cudaGetLastError() != cudaSuccess) return GDR_CUDA_ERROR;
  const bool vec = variant == 0;
  PrepArgs pa{};
  pa.q = static_cast<const __nv_bfloat16*>(q);
  pa.k = static_cast<const __nv_bfloat16*>(k);
  if (l2) {  // the rows' L2 scales (and normalized BF16 copies of q, k, for the backward)
    L2NormArgs la{};
    la.q = pa.q;
    la.k = pa.k;
    la.qn = at<__nv_bfloat16>(base, L.qn);
    la.kn = at<__nv_bfloat16>(base, L.kn);
    la.rq = at<float>(base, L.rq);
    la.rk = at<float>(base, L.rk);
    la.rows = T * Hqk;
    {
      ProfScope ps("l2norm", stream);
      if (launch_l2norm(la, stream) != cudaSuccess) return GDR_CUDA_ERROR;
    }
    // The prep reads the raw q, k and applies the scales in FP32 (the normalized
    // BF16 copies are for the backward's gradient kernel).
    pa.rq = la.rq;
    pa.rk = la.rk;
  }
  pa.v = static_cast<const __nv_bfloat16*>(v);
  pa.g = g;
  pa.beta = beta;
  pa.chunks = chunks;
  pa.Hqk = Hqk;
  pa.HV = HV;
  pa.w = at<__half>(base, L.w);
  pa.u = at<__half>(base, L.u);
  pa.qp = at<__half>(base, L.qp);
  pa.kd = at<__half>(base, L.kd);
  pa.aqk = at<__half>(base, L.aqk);
  pa.gam = at<float>(base, L.gam);
  pa.amat = save_for_bwd ? at<float>(base, L.amat) : nullptr;
  pa.tmat = save_for_bwd ? at<float>(base, L.tmat) : nullptr;
  // Grouped GDN: the tensor-core prep (one CTA per chunk and Q/K head) reads
  // q, k, v through tensor maps.
  PrepTcArgs pt{};
  if (!vec && T > 0) {
    pt.err = device_error_ptr();
    if (!pt.err || !bf16_head_map(&pt.q_map, pa.q, T, Hqk) || !bf16_head_map(&pt.k_map, pa.k, T, Hqk) ||
        !bf16_head_map(&pt.v_map, pa.v, T, HV))
      return GDR_CUDA_ERROR;
  }
  WalkArgs wa{};
  wa.segs = segs;
  wa.HV = HV;
  const bool split = NSEG > N;
  wa.smap = split ? at<float>(base, L.smap) : nullptr;
  wa.sstart = split ? at<float>(base, L.sstart) : nullptr;
  wa.sbias = split ? at<float>(base, L.sbias) : nullptr;
  MergeArgs ma{};
  ma.segs = segs;
  ma.HV = HV;
  ma.smap = wa.smap;
  ma.state = wa.sstart;
  ma.bias = wa.sbias;
  wa.gam = pa.gam;
  wa.err = device_error_ptr();
  if (!wa.err) return GDR_CUDA_ERROR;
  if (NC > 0 && (!fp16_map(&wa.w_map, pa.w, (uint64_t)NC * HV * CH, DK, CH) ||
                 !fp16_map(&wa.kdt_map, pa.kd, (uint64_t)NC * HV * DK, CH, DK) ||
                 !fp16_map(&wa.u_map, pa.u, (uint64_t)NC * HV * CH, DK, CH, LDF) ||
                 !fp16_map(&wa.qp_map, pa.qp, (uint64_t)NC * HV * CH, DK, CH) ||
                 !fp16_map(&wa.aqk_map, pa.aqk, (uint64_t)NC * HV * CH, CH, CH)))
    return GDR_CUDA_ERROR;
  wa.h0 = h0;
  // The state tape and Delta are only kept for a backward.
  wa.tape = save_for_bwd ? at<__nv_bfloat16>(base, L.tape) : nullptr;
  wa.delta = save_for_bwd ? at<float>(base, L.delta) : nullptr;
  wa.ht = ht;
  wa.out = static_cast<__nv_bfloat16*>(out);
  wa.scale = scale;
  // Document groups as in the backward: each group's walk needs only its own
  // prep, so the longest document's walk starts once its chunks are prepared;
  // a pipelined group's walk starts once its first slice is (prep slices on
  // the group's second lane, walk slices on its first).
  wa.carry = at<float>(base, L.fcarry);
  wa.m0 = 0;
  wa.m1 = INT_MAX;
  {
    const int S = slice_chunks();
    bool any_pipe = false;
    for (const DocGroup& G : groups) any_pipe = any_pipe || pipelined(G, S);
    Fork fork(stream, (int)groups.size(), any_pipe);
    if (!fork.begin()) return GDR_CUDA_ERROR;
    auto prep = [&](int64_t c0, int nc, double units, cudaStream_t ls) {
      ProfScope ps("prep", ls, units);
      pa.chunk_base = (int)c0;
      if (vec) return cuda_status(launch_prep(pa, nc, ls));
      pt.p = pa;
      return cuda_status(launch_prep_gdn(pt, nc, ls));
    };
    for (size_t i = 0; i < groups.size() && st == GDR_OK; ++i) {
      const DocGroup& G = groups[i];
      const cudaStream_t ls = fork.lane((int)i);
      const double units = (double)G.tokens * HV;
      const int nsg = (int)(G.s1 - G.s0);
      wa.seg_base = ma.seg_base = (int)G.s0;
      if (pipelined(G, S)) {
        const cudaStream_t lp = fork.lane2((int)i);
        const std::vector<int> sb = slice_bounds((int)(G.c1 - G.c0), S, 2);
        wa.mode = 0;
        for (size_t j = 0; j + 1 < sb.size() && st == GDR_OK; ++j) {
          const int m0 = sb[j], nc = sb[j + 1] - sb[j];
          const double su = (double)std::min<int64_t>((int64_t)nc * CH, G.tokens - (int64_t)m0 * CH) * HV;
          st = prep(G.c0 + m0, nc, su, lp);
          if (st == GDR_OK && !Fork::link(lp, ls)) st = GDR_CUDA_ERROR;
          if (st != GDR_OK) break;
          wa.m0 = m0;
          wa.m1 = m0 + nc;
          ProfScope ps("walk_fwd", ls, su);
          st = cuda_status(launch_walk_fwd_v(wa, nsg, ls));
        }
        wa.m0 = 0;
        wa.m1 = INT_MAX;
        continue;
      }
      st = prep(G.c0, (int)(G.c1 - G.c0), units, ls);
      if (st != GDR_OK) break;
      if (G.split) {
        wa.mode = 1;
        {
          ProfScope ps("walk_fwd_sum", ls, units);
          st = cuda_status(launch_walk_fwd_v(wa, nsg, ls));
        }
        if (st != GDR_OK) break;
        {
          ProfScope ps("merge_fwd", ls, units);
          st = cuda_status(launch_merge(ma, nsg, false, ls));
        }
        if (st != GDR_OK) break;
      }
      wa.mode = 0;
      {
        ProfScope ps("walk_fwd", ls, units);
        st = cuda_status(launch_walk_fwd_v(wa, nsg, ls));
      }
    }
    if (!fork.join() && st == GDR_OK) st = GDR_CUDA_ERROR;
  }
  if (st != GDR_OK) return st;
  if (save_for_bwd) stamp_set(saved, stamp);
  return GDR_OK;
}

gdr_status bwd_impl(int variant, const void* q, const void* k, const void* v, const float* g, const void* beta,
                    const int32_t* cu, const int32_t* cu_host, int32_t N, int64_t T, int32_t Hqk, int32_t HV,
                    float scale, int l2, const void* dout, const float* dht, const void* saved, size_t saved_bytes,
                    void* dq, void* dk, void* dv, float* dg, void* dbeta, float* dh0, void* scratch,
                    size_t scratch_bytes, cudaStream_t stream) {
  if (Hqk <= 0 || HV <= 0 || HV % Hqk != 0) return GDR_INVALID_ARG;
  int64_t NC = 0;
  gdr_status st = plan_host(T, N, cu_host, &NC);
  if (st != GDR_OK) return st;
  if (N == 0) return GDR_OK;
  if (!cu || !saved || !scratch) return GDR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dg || !dbeta)) return GDR_INVALID_ARG;
  if (!aligned_to(q, 16) || !aligned_to(k, 16) || !aligned_to(v, 16) || !aligned_to(g, 16) || !aligned_to(dout, 16) ||
      !aligned_to(dq, 4) || !aligned_to(dk, 4) || !aligned_to(dv, 4))
    return GDR_INVALID_ARG;
  if (!aligned(saved) || !aligned(scratch)) return GDR_INVALID_ARG;
  const int lseg = segment_chunks(N, cu_host, HV);
  std::vector<DocGroup> groups = plan_groups(N, cu_host);
  const int64_t NSEG = assign_segments(groups, N, cu_host, lseg);
  const Layout L = make_layout(T, NC, N, Hqk, HV, l2 != 0, NSEG);
  // A buffer this process filled for other arguments is stale whatever its size.
  Stamp want{T, N, Hqk, HV, variant, lseg, l2 != 0, hash_cu(cu_host, N), 0};
  const StampState known = stamp_check(saved, want, &want.counter);
  if (known == StampState::kMismatch) return GDR_STALE_WORKSPACE;
  if (saved_bytes < L.saved_total || scratch_bytes < L.bwd_total) return GDR_WORKSPACE_TOO_SMALL;
  st = check_device();
  if (st != GDR_OK) return st;
  int* err = device_error_ptr();
  if (!err) return GDR_CUDA_ERROR;
  const bool vec = variant == 0;
  // The backward's own plan (the same tables the forward made), and the
  // device-side check of the saved buffer's header.
  ChunkDesc* chunks = at<ChunkDesc>(scratch, L.bchunks);
  SegDesc* segs = at<SegDesc>(scratch, L.bsegs);
  {
    ProfScope ps("plan", stream);
    k_plan<<<1, 1024, 0, stream>>>(cu, N, std::min(lseg, kNoSplit), at<DocDesc>(scratch, L.bdocs), chunks,
                                   at<int>(scratch, L.border), segs, SavedHeader{}, nullptr);
  }
  {
    ProfScope ps("check", stream);
    k_check_header<<<1, 32, 0, stream>>>(header_of(want), at<SavedHeader>(saved, L.header),
                                         known == StampState::kMatch ? 1 : 0, err);
  }
  if (cudaGetLastError() != cudaSuccess) return GDR_CUDA_ERROR;
  const bool split = NSEG > N;
  WalkBwdArgs wb{};
  wb.segs = segs;
  wb.HV = HV;
  wb.dsend = split ? at<float>(scratch, L.dsend) : nullptr;
  wb.dsbias = split ? at<float>(scratch, L.dsbias) : nullptr;
  MergeArgs mb{};
  mb.segs = segs;
  mb.HV = HV;
  mb.smap = split ? at<float>(saved, L.smap) : nullptr;
  mb.state = wb.dsend;
  mb.bias = wb.dsbias;
  wb.scale = scale;
  const __half* sw = at<__half>(saved, L.w);
  wb.gam = at<float>(saved, L.gam);
  wb.dout = static_cast<const __nv_bfloat16*>(dout);
  wb.dht = dht;
  wb.dstape = at<__nv_bfloat16>(scratch, L.dstape);
  wb.ddelta = at<float>(scratch, L.ddelta);
  wb.dh0 = dh0;
  wb.err = device_error_ptr();
  if (!wb.err) return GDR_CUDA_ERROR;
  if (NC > 0 && (!fp16_map(&wb.w_map, sw, (uint64_t)NC * HV * CH, DK, CH) ||
                 !fp16_map(&wb.kdt_map, at<__half>(saved, L.kd), (uint64_t)NC * HV * DK, CH, DK) ||
                 !fp16_map(&wb.qp_map, at<__half>(saved, L.qp), (uint64_t)NC * HV * CH, DK, CH) ||
                 !fp16_map(&wb.aqk_map, at<__half>(saved, L.aqk), (uint64_t)NC * HV * CH, CH, CH)))
    return GDR_CUDA_ERROR;

  GradStateArgs gs{};
  gs.chunks = chunks;
  gs.HV = HV;
  gs.scale = scale;
  gs.dout = wb.dout;
  gs.tape = at<__nv_bfloat16>(saved, L.tape);
  gs.dstape = wb.dstape;
  gs.delta = at<float>(saved, L.delta);
  gs.ddelta = wb.ddelta;
  gs.dqs = at<float>(scratch, L.dqs);
  gs.dw = at<float>(scratch, L.dw);
  gs.dkd = at<float>(scratch, L.dkd);
  gs.dgam = at<float>(scratch, L.dgam);
  gs.daqk = at<float>(scratch, L.daqk);
  gs.err = wb.err;

  GradArgs ga{};
  // With the in-kernel L2 normalization the gradient kernels read the forward's
  // normalized q, k and produce the gradients of those (dn), which the group
  // reduction maps back to the raw inputs.
  ga.q = l2 ? at<__nv_bfloat16>(saved, L.qn) : static_cast<const __nv_bfloat16*>(q);
  ga.k = l2 ? at<__nv_bfloat16>(saved, L.kn) : static_cast<const __nv_bfloat16*>(k);
  ga.v = static_cast<const __nv_bfloat16*>(v);
  ga.g = g;
  ga.beta = beta;
  ga.dout = wb.dout;
  ga.chunks = chunks;
  ga.Hqk = Hqk;
  ga.HV = HV;
  ga.scale = scale;
  ga.w = sw;
  ga.u = at<__half>(saved, L.u);
  ga.gam = wb.gam;
  ga.delta = gs.delta;
  ga.ddelta = wb.ddelta;
  ga.dqs = gs.dqs;
  ga.dw = gs.dw;
  ga.dkd = gs.dkd;
  ga.dgam = gs.dgam;
  ga.daqk = gs.daqk;
  ga.err = wb.err;
  ga.amat = at<float>(saved, L.amat);
  ga.tmat = at<float>(saved, L.tmat);
  ga.dq = static_cast<__nv_bfloat16*>(dq);
  ga.dk = static_cast<__nv_bfloat16*>(dk);
  ga.dv = static_cast<__nv_bfloat16*>(dv);
  const bool grouped = HV != Hqk || l2;
  ga.dq_part = grouped ? at<float>(scratch, L.dqp) : nullptr;
  ga.dk_part = grouped ? at<float>(scratch, L.dkp) : nullptr;
  ga.dg = dg;
  ga.dbeta = dbeta;
  GroupReduceArgs gr{};
  gr.chunks = chunks;
  gr.Hqk = Hqk;
  gr.HV = HV;
  gr.dq_part = ga.dq_part;
  gr.dk_part = ga.dk_part;
  gr.dq = ga.dq;
  gr.dk = ga.dk;
  gr.q = l2 ? static_cast<const __nv_bfloat16*>(q) : nullptr;
  gr.k = l2 ? static_cast<const __nv_bfloat16*>(k) : nullptr;
  gr.rq = l2 ? at<float>(saved, L.rq) : nullptr;
  gr.rk = l2 ? at<float>(saved, L.rk) : nullptr;

  // Document groups (longest documents first, each on a stream of its own):
  // a group's gradient kernels need only its own walk, so the gradients of the
  // documents whose walks end first run on the SMs the other walks leave idle.
  // Per group: its adjoint walk, then the gradient kernels of its chunks; a
  // pipelined group's walk runs slice by slice (last slice first) on its first
  // lane and each slice's gradient kernels on its second, while the walk goes on.
  wb.carry = at<float>(scratch, L.bcarry);
  wb.m0 = 0;
  wb.m1 = INT_MAX;
  const int S = slice_chunks();
  bool any_pipe = false;
  for (const DocGroup& G : groups) any_pipe = any_pipe || pipelined(G, S);
  Fork fork(stream, (int)groups.size(), any_pipe);
  if (!fork.begin()) return GDR_CUDA_ERROR;
  auto grads = [&](int64_t c0, int nc, double units, cudaStream_t ls) {
    gs.chunk_base = ga.chunk_base = gr.chunk_base = (int)c0;
    gdr_status r;
    {
      ProfScope ps("grad_state", ls, units);
      r = cuda_status(launch_grad_state(gs, nc, ls));
    }
    if (r != GDR_OK) return r;
    {
      ProfScope ps("grad", ls, units);
      r = cuda_status(launch_grad(ga, nc, vec, vec, ls));
    }
    if (r != GDR_OK || !grouped) return r;
    ProfScope ps("group_reduce", ls, units);
    return cuda_status(launch_group_reduce(gr, nc, ls));
  };

  for (size_t i = 0; i < groups.size() && st == GDR_OK; ++i) {
    const DocGroup& G = groups[i];
    const cudaStream_t ls = fork.lane((int)i);
    const double units = (double)G.tokens * HV;
    const int nc = (int)(G.c1 - G.c0), nsg = (int)(G.s1 - G.s0);
    wb.seg_base = mb.seg_base = (int)G.s0;
    if (pipelined(G, S)) {
      const cudaStream_t lg = fork.lane2((int)i);
      wb.mode = 0;
      const std::vector<int> sb = slice_bounds(nc, S, 4);
      for (size_t j = sb.size() - 1; j > 0 && st == GDR_OK; --j) {
        const int m0 = sb[j - 1], sn = sb[j] - sb[j - 1];
        const double su = (double)std::min<int64_t>((int64_t)sn * CH, G.tokens - (int64_t)m0 * CH) * HV;
        wb.m0 = m0;
        wb.m1 = m0 + sn;
        {
          ProfScope ps("walk_bwd", ls, su);
          st = cuda_status(launch_walk_bwd_v(wb, nsg, ls));
        }
        if (st == GDR_OK && !Fork::link(ls, lg)) st = GDR_CUDA_ERROR;
        if (st == GDR_OK) st = grads(G.c0 + m0, sn, su, lg);
      }
      wb.m0 = 0;
      wb.m1 = INT_MAX;
      continue;
    }
    if (G.split) {
      wb.mode = 1;
      {
        ProfScope ps("walk_bwd_sum", ls, units);
        st = cuda_status(launch_walk_bwd_v(wb, nsg, ls));
      }
      if (st != GDR_OK) break;
      {
        ProfScope ps("merge_bwd", ls, units);
        st = cuda_status(launch_merge(mb, nsg, true, ls));
      }
      if (st != GDR_OK) break;
    }
    wb.mode = 0;
    {
      ProfScope ps("walk_bwd", ls, units);
      st = cuda_status(launch_walk_bwd_v(wb, nsg, ls));
    }
    if (st != GDR_OK) break;
    st = grads(G.c0, nc, units, ls);
  }
  if (!fork.join() && st == GDR_OK) st = GDR_CUDA_ERROR;
  if (st != GDR_OK) return st;
  return GDR_OK;
}


// ---------------------------------------------------------------------------
// Fixed device scratch for the no-allocation forward (kda_fwd_noalloc).
// Every GPU that loads this library holds this array until the process exits.
// Host code must not use the symbol itself as a device address: the device
// address is looked up once per device with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up on the
// first call per device; later calls reuse it).  Returns null on failure.
void* static_scratch_ptr(gdr_status* st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *st = GDR_CUDA_ERROR;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
      *st = GDR_CUDA_ERROR;
      return nullptr;
    }
    g_static_ptr[dev] = p;
  }
  *st = GDR_OK;
  return g_static_ptr[dev];
}

}  // namespace
}  // namespace gdr

extern "C" {

const char* gdr_status_string(gdr_status s) {
  switch (s) {
    case GDR_OK: return "GDR_OK";
    case GDR_INVALID_ARG: return "GDR_INVALID_ARG";
    case GDR_BAD_CU_SEQLENS: return "GDR_BAD_CU_SEQLENS";
    case GDR_WORKSPACE_TOO_SMALL: return "GDR_WORKSPACE_TOO_SMALL";
    case GDR_UNSUPPORTED: return "GDR_UNSUPPORTED";
    case GDR_STALE_WORKSPACE: return "GDR_STALE_WORKSPACE";
    case GDR_CUDA_ERROR: return "GDR_CUDA_ERROR";
    case GDR_DEVICE_TIMEOUT: return "GDR_DEVICE_TIMEOUT";
    default: return "GDR_UNKNOWN_STATUS";
  }
}

gdr_status kda_workspace_bytes(int64_t T, int32_t H, int32_t N, const int32_t* cu_seqlens_host, int qk_l2norm,
                               size_t* saved_bytes, size_t* scratch_bytes) {
  return gdr::workspace_bytes(T, H, H, N, cu_seqlens_host, qk_l2norm, saved_bytes, scratch_bytes);
}

gdr_status gdn_workspace_bytes(int64_t T, int32_t Hqk, int32_t HV, int32_t N, const int32_t* cu_seqlens_host,
                               int qk_l2norm, size_t* saved_bytes, size_t* scratch_bytes) {
  return gdr::workspace_bytes(T, Hqk, HV, N, cu_seqlens_host, qk_l2norm, saved_bytes, scratch_bytes);
}

gdr_status kda_fwd(const gdr_bf16* q, const gdr_bf16* k, const gdr_bf16* v, const float* g, const gdr_bf16* beta,
                   const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, int32_t N, int64_t T, int32_t H,
                   float scale, int qk_l2norm, const float* h0, gdr_bf16* out, float* ht, void* saved,
                   size_t saved_bytes, int save_for_bwd, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  return gdr::fwd_impl(0, q, k, v, g, beta, cu_seqlens, cu_seqlens_host, N, T, H, H, scale, qk_l2norm, h0, out, ht,
                       saved, saved_bytes, save_for_bwd, scratch, scratch_bytes, stream);
}

gdr_status kda_bwd(const gdr_bf16* q, const gdr_bf16* k, const gdr_bf16* v, const float* g, const gdr_bf16* beta,
                   const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, int32_t N, int64_t T, int32_t H,
                   float scale, int qk_l2norm, const float* h0, const gdr_bf16* dout, const float* dht,
                   const void* saved, size_t saved_bytes, gdr_bf16* dq, gdr_bf16* dk, gdr_bf16* dv, float* dg,
                   gdr_bf16* dbeta, float* dh0, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  (void)h0;
  return gdr::bwd_impl(0, q, k, v, g, beta, cu_seqlens, cu_seqlens_host, N, T, H, H, scale, qk_l2norm, dout, dht,
                       saved, saved_bytes, dq, dk, dv, dg, dbeta, dh0, scratch, scratch_bytes, stream);
}

gdr_status gdn_fwd(const gdr_bf16* q, const gdr_bf16* k, const gdr_bf16* v, const float* g, const float* beta,
                   const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, int32_t N, int64_t T, int32_t Hqk,
                   int32_t HV, float scale, int qk_l2norm, const float* h0, gdr_bf16* out, float* ht, void* saved,
                   size_t saved_bytes, int save_for_bwd, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  return gdr::fwd_impl(1, q, k, v, g, beta, cu_seqlens, cu_seqlens_host, N, T, Hqk, HV, scale, qk_l2norm, h0, out, ht,
                       saved, saved_bytes, save_for_bwd, scratch, scratch_bytes, stream);
}

gdr_status gdn_bwd(const gdr_bf16* q, const gdr_bf16* k, const gdr_bf16* v, const float* g, const float* beta,
                   const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, int32_t N, int64_t T, int32_t Hqk,
                   int32_t HV, float scale, int qk_l2norm, const float* h0, const gdr_bf16* dout, const float* dht,
                   const void* saved, size_t saved_bytes, gdr_bf16* dq, gdr_bf16* dk, gdr_bf16* dv, float* dg,
                   float* dbeta, float* dh0, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  (void)h0;
  return gdr::bwd_impl(1, q, k, v, g, beta, cu_seqlens, cu_seqlens_host, N, T, Hqk, HV, scale, qk_l2norm, dout, dht,
                       saved, saved_bytes, dq, dk, dv, dg, dbeta, dh0, scratch, scratch_bytes, stream);
}

gdr_status kda_fwd_noalloc(const gdr_bf16* q, const gdr_bf16* k, const gdr_bf16* v, const float* g,
                           const gdr_bf16* beta, const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                           int32_t N, int64_t T, int32_t H, float scale, const float* h0, gdr_bf16* out, float* ht,
                           cudaStream_t stream) {
  size_t need = 0;
  const gdr_status qs = gdr::workspace_bytes(T, H, H, N, cu_seqlens_host, 0, &need, nullptr);
  if (qs != GDR_OK) return qs;
  if (need > gdr::kStaticScratchBytes) return GDR_WORKSPACE_TOO_SMALL;
  if (N == 0) return GDR_OK;
  gdr_status st = GDR_OK;
  void* scratch = gdr::static_scratch_ptr(&st);
  if (!scratch) return st;
  return gdr::fwd_impl(0, q, k, v, g, beta, cu_seqlens, cu_seqlens_host, N, T, H, H, scale, 0, h0, out, ht, nullptr,
                       0, 0, scratch, gdr::kStaticScratchBytes, stream);
}

gdr_status gdr_doc_groups(int32_t N, const int32_t* cu_seqlens_host, int32_t* rank_bounds, int64_t* chunk_bounds,
                          int32_t* n_groups) {
  if (N < 0 || !cu_seqlens_host || !rank_bounds || !chunk_bounds || !n_groups) return GDR_INVALID_ARG;
  if (cu_seqlens_host[0] != 0) return GDR_BAD_CU_SEQLENS;
  for (int32_t n = 0; n < N; ++n)
    if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return GDR_BAD_CU_SEQLENS;
  if (N == 0) {
    *n_groups = 0;
    return GDR_OK;
  }
  const std::vector<gdr::DocGroup> g = gdr::plan_groups(N, cu_seqlens_host);
  *n_groups = (int32_t)g.size();
  for (size_t i = 0; i < g.size(); ++i) {
    rank_bounds[i] = g[i].r0;
    rank_bounds[i + 1] = g[i].r1;
    chunk_bounds[i] = g[i].c0;
    chunk_bounds[i + 1] = g[i].c1;
  }
  return GDR_OK;
}

gdr_status gdr_segment_plan(int32_t N, const int32_t* cu_seqlens_host, int32_t HV, int32_t* seg_chunks,
                            int64_t* n_segments) {
  if (N < 0 || !cu_seqlens_host || HV <= 0 || !seg_chunks || !n_segments) return GDR_INVALID_ARG;
  if (cu_seqlens_host[0] != 0) return GDR_BAD_CU_SEQLENS;
  for (int32_t n = 0; n < N; ++n)
    if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return GDR_BAD_CU_SEQLENS;
  if (N == 0) {
    *seg_chunks = 0;
    *n_segments = 0;
    return GDR_OK;
  }
  const int lseg = gdr::segment_chunks(N, cu_seqlens_host, HV);
  std::vector<gdr::DocGroup> groups = gdr::plan_groups(N, cu_seqlens_host);
  *n_segments = gdr::assign_segments(groups, N, cu_seqlens_host, lseg);
  *seg_chunks = lseg >= gdr::kNoSplit ? 0 : lseg;
  return GDR_OK;
}

gdr_status gdr_walk_slices(int32_t nchunks, int32_t direction, int32_t* bounds, int32_t cap, int32_t* n_slices) {
  if (!bounds || !n_slices || nchunks < 0 || (direction != 0 && direction != 1) || cap < 1) return GDR_INVALID_ARG;
  if (nchunks == 0) {
    bounds[0] = 0;
    *n_slices = 0;
    return GDR_OK;
  }
  const std::vector<int> b = gdr::slice_bounds(nchunks, gdr::slice_chunks(), direction ? 4 : 2);
  if ((int64_t)b.size() > cap) return GDR_INVALID_ARG;
  for (size_t i = 0; i < b.size(); ++i) bounds[i] = b[i];
  *n_slices = (int32_t)b.size() - 1;
  return GDR_OK;
}

gdr_status gdr_inject_device_error(int code) {
  if (code <= 0) return GDR_INVALID_ARG;
  int* p = gdr::device_error_ptr();
  if (!p) return GDR_CUDA_ERROR;
  return cudaMemcpy(p, &code, sizeof(int), cudaMemcpyHostToDevice) == cudaSuccess ? GDR_OK : GDR_CUDA_ERROR;
}

gdr_status gdr_selftest_wait(uint64_t limit_ns, cudaStream_t stream) {
  if (limit_ns < 1 || limit_ns > 100000000ull) return GDR_INVALID_ARG;
  int* p = gdr::device_error_ptr();
  if (!p) return GDR_CUDA_ERROR;
  gdr::k_selftest_wait<<<1, 32, 0, stream>>>(limit_ns, p);
  return gdr::cuda_status(cudaGetLastError());
}

gdr_status gdr_check_device(void) {
  int* p = gdr::device_error_ptr();
  if (!p) return GDR_CUDA_ERROR;
  if (cudaDeviceSynchronize() != cudaSuccess) return GDR_CUDA_ERROR;
  int code = 0;
  if (cudaMemcpy(&code, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GDR_CUDA_ERROR;
  if (code != 0) {
    const int zero = 0;
    cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return code == gdr::kStaleCode ? GDR_STALE_WORKSPACE : GDR_DEVICE_TIMEOUT;
  }
  return GDR_OK;
}

uint64_t gdr_launch_count(void) { return gdr::g_launches.load(); }

int gdr_set_serial(int on) { return gdr::g_serial.exchange(on != 0) ? 1 : 0; }

int gdr_set_segment_chunks(int chunks) { return gdr::g_seg_chunks.exchange(chunks > 0 ? chunks : 0); }

int gdr_set_slice_chunks(int chunks) {
  return gdr::g_slice_chunks.exchange(chunks > 0 ? std::max(2, chunks & ~1) : 0);
}

int gdr_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(gdr::g_prof_mu);
  if (on) gdr::prof_clear_locked();
  gdr::g_prof_on = on != 0;
  return GDR_OK;
}

gdr_status gdr_profile_report(char* buf, size_t buf_bytes) {
  std::lock_guard<std::mutex> lk(gdr::g_prof_mu);
  struct Agg {
    int n = 0;
    double ms = 0, units = 0;
  };
  std::map<std::string, Agg> agg;
  std::vector<std::string> order;
  for (auto& r : gdr::g_prof) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return GDR_CUDA_ERROR;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return GDR_CUDA_ERROR;
    if (agg.find(r.name) == agg.end()) order.push_back(r.name);
    Agg& a = agg[r.name];
    a.n += 1;
    a.ms += ms;
    a.units += r.units;
  }
  std::string out;
  for (auto& n : order) {
    char line[200];
    std::snprintf(line, sizeof(line), "%s %d %.6f %.0f\n", n.c_str(), agg[n].n, agg[n].ms, agg[n].units);
    out += line;
  }
  if (!buf || buf_bytes < out.size() + 1) return GDR_INVALID_ARG;
  std::memcpy(buf, out.c_str(), out.size() + 1);
  return GDR_OK;
}

}  // extern "C"
