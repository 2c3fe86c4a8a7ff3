// Shared definitions of the GDN library: sizes, the workspace layout and the planner.
//
// The planner turns cu_seqlens / init_idx into
//   * the chunk map: every document is cut into 64-token chunks starting at its own first
//     token, the last chunk of a document may be partial ("Musings on long-context
//     fine-tuning", section "Isolating the recurrent layers": the state restarts at every
//     cu_seqlens boundary; "How to Speed Up GDN Kernels for Qwen Models", section "What GDN
//     actually computes": chunks of 64 tokens);
//   * the segment map: when documents x value heads cannot fill the SMs, long documents are
//     cut into segments of L chunks that run in parallel ("The real enemy: an idle GPU" and
//     "Lever 1: the gate is also a license to parallelize" on the same page);
//   * each segment's dependency: the start state is known at launch (zero or a pool entry),
//     or it is the end state of the previous segment, or the final state of another document
//     of the same call (a fork).
// The same functions run on the host (gdn_plan_host, tests) and on the device (plan kernel),
// so the two produce identical maps.
#pragma once
#include <cstddef>
#include <cstdint>

#ifdef __CUDACC__
#define GDN_HD __host__ __device__ __forceinline__
#else
#define GDN_HD inline
#endif

namespace gdn {

constexpr int kChunk = 64;        // tokens per chunk
constexpr int kDim = 128;         // d_k = d_v
constexpr int kMinSegChunks = 4;  // shortest automatic segment (chunks)
// Per-token factors of the inference chain per (chunk, value head): e^{gamma_C - gamma_t} (t < 64),
// the output factor of token t (64 + t), e^{gamma_C} (128); 144 floats keep records 16-byte aligned.
constexpr int kFacFloats = 144;

// q and k normalisation (GDN_FLAG_L2NORM_QK): y = x (x . x + kL2NormEps)^{-1/2} per row of 128.
constexpr float kL2NormEps = 1e-6f;
// Option flags that change the inputs (mirror include/gdn.h).
constexpr int kFlagL2Norm = 8, kFlagFp16 = 16;

// Workspace copies of the inputs, placed after the forward's or the backward's layout: with
// GDN_FLAG_L2NORM_QK and/or GDN_FLAG_FP16_INPUTS, q' and k' (bf16 [T][Hk][128], normalised and/or
// converted); with fp16 inputs also v' and, in a backward workspace, dout' (bf16 [T][Hv][128]).
struct InputCopies {
  size_t q, k, v, dout, total;  // byte offsets from the start of the region, and its size
};
inline InputCopies input_copies(int T, int Hk, int Hv, int flags, bool bwd) {
  InputCopies c{0, 0, 0, 0, 0};
  if (!(flags & (kFlagL2Norm | kFlagFp16))) return c;
  const size_t qk = (size_t)T * Hk * kDim * 2, vv = (size_t)T * Hv * kDim * 2;
  c.k = qk;
  c.v = 2 * qk;
  c.dout = 2 * qk + ((flags & kFlagFp16) ? vv : 0);
  c.total = c.dout + ((flags & kFlagFp16) && bwd ? vv : 0);
  c.total = (c.total + 255) / 256 * 256;
  return c;
}

// Status codes (mirror include/gdn.h).
constexpr int kOk = 0, kErrInvalid = -1, kErrUnsupported = -2, kErrCuda = -3, kErrTimeout = -4,
              kErrWorkspace = -5;

// Segment dependency encoding (seg_info[4 * s + 3]).
//   -1        start state known at launch (zero or a pool entry)
//   s' >= 0   end state of segment s' (the previous segment of the same document)
//   <= -2     final state of document j = -dep - 2 (fork)
GDN_HD int dep_fork_seq(int dep) { return -dep - 2; }

struct Header {
  int32_t status;      // first device-side error (0 = ok)
  int32_t n_chunks;    // chunks in this call
  int32_t n_segs;      // segments in this call
  int32_t seg_chunks;  // chosen segment length (chunks); 0 = no split
  int32_t n_p1;        // pass-1 units (segment, part)
  uint32_t q_p1;       // work-queue tickets
  uint32_t q_chain;
  int32_t n_walk;      // pass-1 walks (documents whose known-start first segment has middle segments)
  int32_t pad[56];
};
static_assert(sizeof(Header) == 256, "header is 256 bytes");

struct PlanDims {
  int N, T, Hk, Hv, n_init;
  int num_sms;
  int seg_override;  // options.segment_chunks
  int mode;          // 0 exact, 1 truncate
};

GDN_HD int64_t max_chunks(int N, int T) { return (int64_t)T / kChunk + N + 1; }

// Upper bound on segments that get a slot (published end state / pass-1 matrices).
GDN_HD int64_t max_split_segs(const PlanDims& d) {
  const int64_t cmax = max_chunks(d.N, d.T);
  if (d.seg_override < 0) return 0;
  if (d.seg_override > 0) return (int64_t)d.N + cmax / d.seg_override + 1;
  if ((int64_t)d.N * d.Hv >= 2LL * d.num_sms) return 0;
  return (int64_t)d.N + (d.num_sms + d.Hv - 1) / d.Hv + 1;
}
GDN_HD int64_t max_segs(const PlanDims& d) { return (int64_t)d.N + max_split_segs(d) + 1; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Forward workspace layout (byte offsets from the workspace base).
struct FwdLayout {
  size_t header, seq_chunk0, seq_seg0, chunk_seq, chunk_tok0, chunk_len, seg_info, seg_slot, p1_list, walk_list;
  size_t flags_seg, flags_fin, flags_p1, walk_ctr, mzero, gam, fac, contr, tw, tu, pimg, pub, mmat, bmat, mimg, total;
  int64_t cmax, smax, slots;
};

inline FwdLayout fwd_layout(const PlanDims& d) {
  FwdLayout L{};
  L.cmax = max_chunks(d.N, d.T);
  L.smax = max_segs(d);
  L.slots = max_split_segs(d);
  const size_t state = (size_t)kDim * kDim * sizeof(float);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  L.header = take(sizeof(Header));
  L.seq_chunk0 = take(sizeof(int32_t) * (d.N + 1));
  L.seq_seg0 = take(sizeof(int32_t) * (d.N + 1));
  L.chunk_seq = take(sizeof(int32_t) * L.cmax);
  L.chunk_tok0 = take(sizeof(int32_t) * L.cmax);
  L.chunk_len = take(sizeof(int32_t) * L.cmax);
  L.seg_info = take(sizeof(int32_t) * 4 * L.smax);
  L.seg_slot = take(sizeof(int32_t) * L.smax);
  L.p1_list = take(sizeof(int32_t) * 2 * (2 * L.slots + 1));
  L.walk_list = take(sizeof(int32_t) * (L.slots + 1));
  L.flags_seg = take(sizeof(int32_t) * (size_t)L.smax * d.Hv);
  L.flags_fin = take(sizeof(int32_t) * (size_t)(d.N + 1) * d.Hv);
  L.flags_p1 = take(sizeof(int32_t) * ((size_t)L.slots * d.Hv + 1));  // a segment's M and B are written
  // per (document, value head): pass-1 units that compute a transition M and a local end state B,
  // and units that have decided (the first count is final once the second is complete)
  L.walk_ctr = take(sizeof(int32_t) * 2 * (size_t)(d.N + 1) * d.Hv);
  L.mzero = take(sizeof(int32_t) * ((size_t)L.slots * d.Hv + 1));
  L.gam = take(sizeof(float) * (size_t)L.cmax * d.Hv * kChunk);
  L.fac = take(sizeof(float) * (size_t)L.cmax * d.Hv * kFacFloats);
  L.contr = take(sizeof(int32_t) * (size_t)L.cmax * d.Hv);
  L.tw = take((size_t)L.cmax * d.Hv * kChunk * kChunk * 2);
  L.tu = take((size_t)L.cmax * d.Hv * kChunk * kChunk * 2);
  L.pimg = take((size_t)L.cmax * d.Hv * kChunk * kChunk * 2);
  L.pub = take(state * (size_t)L.slots * d.Hv);
  const bool exact = d.mode == 0;
  L.mmat = take(exact ? state * (size_t)L.slots * d.Hv : 0);
  L.bmat = take(exact ? state * (size_t)L.slots * d.Hv : 0);
  L.mimg = take(exact ? state * (size_t)L.slots * d.Hv : 0);  // M as compensated bf16 operand images
  L.total = o;
  return L;
}

// ------------------------------------------------------------------------------ planner pieces

// Validation of one document i (0 <= i < N). Returns 0 or kErrInvalid.
GDN_HD int plan_check_doc(int i, const int32_t* cu, const int32_t* init_idx, int n_init) {
  if (cu[i + 1] < cu[i]) return kErrInvalid;
  if (init_idx) {
    const int x = init_idx[i];
    if (x < -1) return kErrInvalid;
    if (x >= n_init && x - n_init >= i) return kErrInvalid;
  }
  return kOk;
}

// fp32 64x64 scratch layout shared by the gradient kernels and the T records of kkt_solve:
// element (i, j) at i*64 + 4*((j/4 XOR i) mod 16) + j mod 4. Sixteen threads that each own a row
// and read the same column hit distinct 16-byte granules (at most two to a bank), and a warp that
// reads a row (consecutive j) stays conflict-free; 4-element groups stay contiguous and aligned.
GDN_HD int fz(int i, int j) { return i * 64 + ((((j >> 2) ^ i) & 15) << 2) + (j & 3); }

GDN_HD int doc_chunks(int i, const int32_t* cu) { return (cu[i + 1] - cu[i] + kChunk - 1) / kChunk; }

// Segment length in chunks (0 = no split) from the totals of this call.
GDN_HD int plan_seg_len(const PlanDims& d, int total_chunks, int longest_doc_chunks) {
  if (d.seg_override < 0) return 0;
  if (d.seg_override > 0) return longest_doc_chunks > d.seg_override ? d.seg_override : 0;
  if ((int64_t)d.N * d.Hv >= 2LL * d.num_sms) return 0;
  // Aim at about one (segment, head) chain per SM: L = total chunks * heads / SMs, floored at
  // kMinSegChunks ("Lever 1": segment length balances sequential depth against parallel width).
  int64_t L = ((int64_t)total_chunks * d.Hv + d.num_sms - 1) / d.num_sms;
  if (L < kMinSegChunks) L = kMinSegChunks;
  return longest_doc_chunks > L ? (int)L : 0;
}

GDN_HD int doc_segs(int nch, int L) { return (L > 0 && nch > L) ? (nch + L - 1) / L : 1; }

// Last index i in [0, n) with off[i] <= x (off nondecreasing, off[0] <= x).
GDN_HD int upper_index(const int32_t* off, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Chunk entry c: sequence, first token, length. seq_chunk0 has N+1 entries.
GDN_HD void plan_chunk(int c, const int32_t* seq_chunk0, int N, const int32_t* cu, int32_t* seq, int32_t* tok0,
                       int32_t* len) {
  // The document owning chunk c is the last i with seq_chunk0[i] <= c among documents that
  // have chunks; empty documents share their offset with the next one, so take the last.
  const int i = upper_index(seq_chunk0, N, c);
  const int t0 = cu[i] + (c - seq_chunk0[i]) * kChunk;
  const int e = cu[i + 1];
  *seq = i;
  *tok0 = t0;
  *len = (e - t0) < kChunk ? (e - t0) : kChunk;
}

// Segment entry s: info[0..3] = sequence, first chunk, chunk count, dependency.
GDN_HD void plan_segment(int s, const int32_t* seq_seg0, const int32_t* seq_chunk0, int N, const int32_t* cu,
                         int L, const int32_t* init_idx, int n_init, int32_t* info) {
  const int i = upper_index(seq_seg0, N, s);
  const int k = s - seq_seg0[i];
  const int nch = doc_chunks(i, cu);
  const int nseg = doc_segs(nch, L);
  int first = 0, cnt = nch;
  if (nseg > 1) {
    first = k * L;
    cnt = (nch - first) < L ? (nch - first) : L;
  }
  info[0] = i;
  info[1] = seq_chunk0[i] + first;
  info[2] = cnt;
  if (k > 0) {
    info[3] = s - 1;
  } else {
    const int x = init_idx ? init_idx[i] : -1;
    info[3] = (x >= n_init) ? -(x - n_init) - 2 : -1;
  }
}

}  // namespace gdn
