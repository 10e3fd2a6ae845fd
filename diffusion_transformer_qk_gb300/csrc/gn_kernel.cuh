// Group norm + SiLU kernels for sm_103a ("fused qknorm rope Flux 2.0",
// section "Not in this PR — follow-ups": group_norm_silu for the VAE).
//
// Activations are NCHW, so the (C/G)*H*W elements of sample n, group g are
// one contiguous span.  A group has few and large spans (32 groups of up to
// millions of elements in a VAE decoder), so each span is cut into P pieces.
// Per piece: its count, its mean relative to the span's shift K (the lower
// median of the span's first 8 values) and its sum of squared deviations
// (moments.cuh: each thread's part from fp32 sums around its own first
// element, merged in an xor tree in each warp, the warps' parts merged in
// order).  Per span: the P pieces' parts
// merged pairwise in one fixed order (combine_span) into m1 (the mean is
// K + m1) and var, then per channel a = gamma[c] * rstd, b = beta[c] -
// m1 * a, y = (x - K)*a + b and out = silu(y) = y / (1 + exp(-y)).
// (exp and the reciprocal on the special-function unit: ex2.approx and
// rcp.approx, about 2 ulp.)
//
// Two paths, with the same arithmetic (equal bits for equal pieces):
//   two-pass: gn_stats_kernel (one CTA per piece) writes the pieces' sums
//     to the workspace, gn_apply_kernel (one CTA per piece) combines and
//     writes; x is read twice and no CTA waits for another.
//   fused: gn_fused_kernel, one persistent launch that reads x once (see
//     the comment above it).
//
// Workspace records, 16 bytes per piece and one more per span: two 8-byte
// words, each (tag << 32) | the bits of an fp32 value: (mean - K, sum of
// squared deviations) for piece i < P, (K, 0) at index P.  An 8-byte store is single-copy atomic, so a
// word that carries the expected tag also carries its value: the fused
// path's waits look for its per-call tag, with no counter and no fence.
// The two-pass path writes tag 0 and does not look at tags.
#pragma once

#include "moments.cuh"
#include "qknr_ptx.cuh"

namespace qknr {

constexpr int kGnThreads = 256;
constexpr int kGnWarps = kGnThreads / 32;
constexpr int kGnBatch = 8;          // 16-byte loads a thread keeps in flight
constexpr int kGnCoefFloats = 4;     // per span: m1, rstd, K (and one float of padding)

struct GnParams {
  const char* x;
  char* out;
  const float* gamma;
  const float* beta;
  unsigned long long* rec;     // [spans][pieces + 1][2] tagged words
  long long span_len;          // L = (C/G) * H * W elements
  long long hw;                // H * W (a multiple of 8)
  long long piece_len;         // elements per piece (a multiple of 8)
  int channels;                // C
  int groups;                  // G
  int group_channels;          // C / G
  int pieces;                  // P pieces per span
  int span0;                   // first span (n*G + g) of this launch
  float eps;
  int* status;                 // checked builds: QKNR_ERR_BOUNDS goes here
  // address spans of the buffers (checked builds test every access against them)
  MemSpan sp_x, sp_out, sp_ws, sp_gamma, sp_beta;
};

__device__ __forceinline__ unsigned long long tagged(unsigned tag, float v) {
  return (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(v);
}

__device__ __forceinline__ float tagged_value(unsigned long long w) {
  return __uint_as_float(static_cast<unsigned>(w));
}

__device__ __forceinline__ unsigned tag_of(unsigned long long w) { return static_cast<unsigned>(w >> 32); }

// 16-byte record store / load at gpu scope, each 8-byte half single-copy atomic
__device__ __forceinline__ void st_record(unsigned long long* p, unsigned long long a, unsigned long long b) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

__device__ __forceinline__ ulonglong2 ld_record(const unsigned long long* p) {
  unsigned long long a, b;
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
  return make_ulonglong2(a, b);
}

// The part of one piece (moments.cuh) from the threads' parts: an xor tree
// in each warp, then thread 0 merges the warps' parts in order (warp w
// covers vectors tid, tid + kGnThreads, ... of the piece's nvec 16-byte
// vectors for its lanes tid).  `red` holds 2 * kGnWarps floats; `sync` is
// the barrier over the kGnThreads threads.  Valid in thread 0.
template <typename Sync>
__device__ __forceinline__ Moments piece_moments(const Moments& mine, int nvec, float* red, Sync sync) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Moments wp = warp_moments(mine, warp_count(warp, nvec, kGnThreads, 8));
  if (lane == 0) {
    red[warp] = wp.u;
    red[kGnWarps + warp] = wp.m;
  }
  sync();
  Moments t{0.0f, 0.0f, 0.0f};
  if (threadIdx.x == 0) {
    const float r = red[0];                      // warp 0 holds values whenever the piece does
    RefSums sums;
    for (int w = 0; w < kGnWarps; ++w) sums.add(Moments{warp_count(w, nvec, kGnThreads, 8), red[w], red[kGnWarps + w]}, r);
    t = merged(8.0f * static_cast<float>(nvec), r, sums);
  }
  return t;
}

// Bounded-wait context of the fused path's record polls.
struct RecordWait {
  unsigned tag;                      // the call's tag
  unsigned long long limit_ns;
  volatile int* abort_cta;           // shared-memory abort flag of the CTA
  unsigned* abort_grid;              // == tag once any CTA has given up
  int* status;
};

// whether this CTA or another has given up (then this CTA's flag is raised)
__device__ __forceinline__ bool grid_aborted(const RecordWait& w) {
  if (*w.abort_cta) return true;
  if (*reinterpret_cast<volatile unsigned*>(w.abort_grid) != w.tag) return false;
  *w.abort_cta = 1;
  return true;
}

__device__ __forceinline__ void give_up(const RecordWait& w) {
  *w.abort_cta = 1;
  atomicExch(w.abort_grid, w.tag);
  if (w.status) atomicCAS(w.status, 0, kStatusTimeout);
}

// Mean and 1/sqrt(var + eps) of a span from its records, in one fixed
// order: lane l sums pieces l, l+32, l+64, ... around the mean of its first
// one (up to eight records in flight; the order of the additions does not
// change), then the lanes' parts are merged by an xor tree (moments.cuh);
// with m1 the mean relative to K, var = m / L.  Pieces hold
// piece_len elements, the last one the rest of the span.  Called by one
// whole warp; lane 0 writes coef[0] = m1, coef[1] = rstd and coef[2] = K
// (kGnCoefFloats floats).
//
// kWait (fused path): a record counts only once both its words carry
// w->tag; a lane re-reads from its first record without it, so the records
// are polled and read in the same loads.  Returns false, in every lane,
// when a lane gave up (bounded by w->limit_ns, or another CTA gave up).
template <bool kWait>
__device__ __forceinline__ bool combine_span(const unsigned long long* rec, int pieces, long long span_len,
                                             long long piece_len, float eps, const RecordWait* w, float* coef,
                                             const MemSpan& ws, int* status) {
  constexpr int kBatch = 8;
  const int lane = threadIdx.x & 31;
  // checked builds: the span's P + 1 records inside the workspace
  if (!in_span(rec, static_cast<unsigned long long>(pieces + 1) * 16, ws, status)) return false;
  // the shift K (written with piece 0's sums), loaded with the first batch
  unsigned long long kw = lane == 0 ? ld_record(rec + 2 * pieces).x : 0ull;
  float nl = 0.0f, rl = 0.0f;                        // this lane's count and reference
  RefSums sl;
  const float full_n = static_cast<float>(piece_len);
  const float last_n = static_cast<float>(span_len - static_cast<long long>(pieces - 1) * piece_len);
  bool ok = true;
  unsigned long long t0 = 0;
  unsigned backoff = 32;                             // ns between polls, doubling to 1 us
  int i = lane;
  while (i < pieces) {
    ulonglong2 v[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int k = i + 32 * b;
      v[b] = k < pieces ? ld_record(rec + 2 * k) : make_ulonglong2(0ull, 0ull);
    }
    int took = 0;
    bool stop = false;
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (!stop && i + 32 * b < pieces && (!kWait || (tag_of(v[b].x) == w->tag && tag_of(v[b].y) == w->tag))) {
        const int k = i + 32 * b;
        const Moments pc{k == pieces - 1 ? last_n : full_n, tagged_value(v[b].x), tagged_value(v[b].y)};
        if (nl == 0.0f) rl = pc.u;
        sl.add(pc, rl);
        nl = __fadd_rn(nl, pc.n);
        ++took;
      } else {
        stop = true;
      }
    }
    i += 32 * took;
    if (kWait && took == 0) {
      if (t0 == 0) t0 = global_timer_ns();
      if (grid_aborted(*w)) {
        ok = false;
        break;
      }
      if (global_timer_ns() - t0 > w->limit_ns) {
        give_up(*w);
        ok = false;
        break;
      }
      __nanosleep(backoff);
      backoff = backoff < 1024 ? 2 * backoff : 1024;
    } else {
      backoff = 32;
    }
  }
  if (kWait && lane == 0 && ok) {
    if (t0 == 0) t0 = global_timer_ns();
    while (tag_of(kw) != w->tag) {
      if (grid_aborted(*w)) {
        ok = false;
        break;
      }
      if (global_timer_ns() - t0 > w->limit_ns) {
        give_up(*w);
        ok = false;
        break;
      }
      __nanosleep(backoff);
      backoff = backoff < 1024 ? 2 * backoff : 1024;
      kw = ld_record(rec + 2 * pieces).x;
    }
  }
  if (!__all_sync(0xffffffffu, ok)) return false;
  const Moments acc = warp_moments(merged(nl, rl, sl), static_cast<float>(span_len));
  if (lane == 0) {
    const float var = __fmul_rn(acc.m, __frcp_rn(static_cast<float>(span_len)));
    coef[0] = acc.u;
    coef[1] = rsqrtf(__fadd_rn(var, eps));
    coef[2] = tagged_value(kw);
  }
  return true;
}

// Folded coefficients of channel c for x - K: a = gamma[c] * rstd and
// b = beta[c] - m1 * a, so y = (x - K) * a + b.  Folding the whole mean
// into b instead (y = x * a + b) would make y the difference of two fp32
// terms of size |mean| * a, whose rounding costs several ulps of a small y
// when |mean| is large against the spread; x - K is exact for nearby
// values and m1 is small.
__device__ __forceinline__ void fold_channel(float g, float be, float m1, float rstd, float2& A, float2& B) {
  const float a = __fmul_rn(g, rstd);
  const float bb = __fmaf_rn(-m1, a, be);
  A = make_float2(a, a);
  B = make_float2(bb, bb);
}

// Channel (within the group) of element e of a span: e < L < 2^31
__device__ __forceinline__ unsigned channel_of(long long e, long long hw) {
  return static_cast<unsigned>(e) / static_cast<unsigned>(hw);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// silu((x - K)*a + b) of one 16-byte vector (a vector never straddles a
// channel: H*W is a multiple of 8), NK = (-K, -K): y = (x - K)*a + b, e^-y = 2^(-y * log2(e)) on the
// special-function unit, silu(y) = y * (1 / (1 + e^-y)), the fp32 steps on
// paired instructions.  Saturates correctly: e^-y overflows to +inf for very
// negative y, giving y * 0.
constexpr float kNegLog2e = -1.4426950408889634f;    // -log2(e)

template <typename T>
__device__ __forceinline__ uint4 silu_affine(const uint4& raw, const float2& NK, const float2& A, const float2& B) {
  float2 X[4], O[4];
  Elem<T>::unpack(raw, X);
  const float2 nl = make_float2(kNegLog2e, kNegLog2e), one = make_float2(1.0f, 1.0f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 y = __ffma2_rn(__fadd2_rn(X[j], NK), A, B);
    const float2 t = __fmul2_rn(y, nl);
    const float2 d = __fadd2_rn(make_float2(ex2_approx(t.x), ex2_approx(t.y)), one);
    O[j] = __fmul2_rn(y, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
  }
  return Elem<T>::pack(O);
}

struct CtaSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

template <typename T>
__global__ void __launch_bounds__(kGnThreads) gn_stats_kernel(const __grid_constant__ GnParams p) {
  __shared__ float red[2 * kGnWarps];
  const int span = p.span0 + blockIdx.y;
  const int piece = blockIdx.x;
  const char* base = p.x + static_cast<long long>(span) * p.span_len * 2;
  const long long lo = static_cast<long long>(piece) * p.piece_len;
  long long hi = lo + p.piece_len;
  if (hi > p.span_len) hi = p.span_len;
  // checked builds: the span inside x, its records inside the workspace
  // (the same answer in every thread of the block)
  if (!in_span(base, static_cast<unsigned long long>(p.span_len) * 2, p.sp_x, p.status) ||
      !in_span(p.rec + static_cast<long long>(span) * (p.pieces + 1) * 2, static_cast<unsigned long long>(p.pieces + 1) * 16,
               p.sp_ws, p.status))
    return;
  float2 first[4];
  Elem<T>::unpack(__ldg(reinterpret_cast<const uint4*>(base)), first);
  const float K = shift_of_first8(first);
  // this thread's vectors are tid, tid + kGnThreads, ... of the piece's
  // nvec, in batches of kGnBatch; each batch is a part, summed around the
  // first value of its first vector (so a large value holds down the
  // precision of at most its batch), and the parts are merged around the
  // first one.  A piece of at most kGnBatch vectors per thread is one batch,
  // the fused kernel's stats warps' part.
  const int nvec = static_cast<int>((hi - lo) / 8);
  float tn = 0.0f, tr = 0.0f;
  RefSums ts;
  // kGnBatch independent 16-byte loads in flight per thread before any is used
  constexpr long long kStride = kGnThreads * 8;
  for (long long e0 = lo + threadIdx.x * 8; e0 < hi; e0 += kStride * kGnBatch) {
    uint4 v[kGnBatch];
#pragma unroll
    for (int b = 0; b < kGnBatch; ++b) {
      const long long e = e0 + b * kStride;
      v[b] = e < hi ? __ldg(reinterpret_cast<const uint4*>(base + e * 2)) : make_uint4(0, 0, 0, 0);
    }
    float2 f[4];
    Elem<T>::unpack(v[0], f);
    const float kb = f[0].x;
    const float2 nk = make_float2(-kb, -kb);
    float2 a1 = make_float2(0.0f, 0.0f), a2 = make_float2(0.0f, 0.0f);
    float nb = 0.0f;
#pragma unroll
    for (int b = 0; b < kGnBatch; ++b) {
      if (e0 + b * kStride < hi) {
        float2 X[4];
        Elem<T>::unpack(v[b], X);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 d = __fadd2_rn(X[j], nk);
          a1 = __fadd2_rn(a1, d);
          a2 = __ffma2_rn(d, d, a2);
        }
        nb = __fadd_rn(nb, 8.0f);
      }
    }
    const Moments bp = moments_of(nb, __fsub_rn(kb, K), __fadd_rn(a1.x, a1.y), __fadd_rn(a2.x, a2.y));
    if (tn == 0.0f) tr = bp.u;
    ts.add(bp, tr);
    tn = __fadd_rn(tn, nb);
  }
  const Moments mine = tn == 0.0f ? Moments{0.0f, 0.0f, 0.0f} : merged(tn, tr, ts);
  const Moments pm = piece_moments(mine, nvec, red, CtaSync());
  if (threadIdx.x == 0) {
    unsigned long long* rec = p.rec + static_cast<long long>(span) * (p.pieces + 1) * 2;
    st_record(rec + 2 * piece, tagged(0u, pm.u), tagged(0u, pm.m));
    // the shift, kept here because an in-place apply overwrites x
    if (piece == 0) st_record(rec + 2 * p.pieces, tagged(0u, K), tagged(0u, 0.0f));
  }
}

template <typename T>
__global__ void __launch_bounds__(kGnThreads) gn_apply_kernel(const __grid_constant__ GnParams p) {
  __shared__ float coef[kGnCoefFloats];      // m1, 1/sqrt(var + eps) and K of the span
  const int span = p.span0 + blockIdx.y;
  const int piece = blockIdx.x;
  const char* base = p.x + static_cast<long long>(span) * p.span_len * 2;
  char* obase = p.out + static_cast<long long>(span) * p.span_len * 2;
  // checked builds: the span inside x and out (the same in every thread)
  if (!in_span(base, static_cast<unsigned long long>(p.span_len) * 2, p.sp_x, p.status) ||
      !in_span(obase, static_cast<unsigned long long>(p.span_len) * 2, p.sp_out, p.status))
    return;
  if (threadIdx.x < 32)
    combine_span<false>(p.rec + static_cast<long long>(span) * (p.pieces + 1) * 2, p.pieces, p.span_len,
                        p.piece_len, p.eps, nullptr, coef, p.sp_ws, p.status);
  __syncthreads();
  const float m1 = coef[0], rstd = coef[1];
  const float2 nk = make_float2(-coef[2], -coef[2]);
  const int ch0 = (span % p.groups) * p.group_channels;
  const long long lo = static_cast<long long>(piece) * p.piece_len;
  long long hi = lo + p.piece_len;
  if (hi > p.span_len) hi = p.span_len;
  long long ch_end = -1;
  float2 A = make_float2(0.0f, 0.0f), B = make_float2(0.0f, 0.0f);
  constexpr long long kStride = kGnThreads * 8;
  for (long long e0 = lo + threadIdx.x * 8; e0 < hi; e0 += kStride * kGnBatch) {
    // plain loads (with out == x this kernel writes what it reads), all in
    // flight before the first is used
    uint4 v[kGnBatch];
#pragma unroll
    for (int b = 0; b < kGnBatch; ++b) {
      const long long e = e0 + b * kStride;
      v[b] = e < hi ? *reinterpret_cast<const uint4*>(base + e * 2) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int b = 0; b < kGnBatch; ++b) {
      const long long e = e0 + b * kStride;
      if (e >= hi) break;
      if (e >= ch_end) {
        const unsigned cl = channel_of(e, p.hw);
        ch_end = (static_cast<long long>(cl) + 1) * p.hw;
        const float* gp = p.gamma + ch0 + cl;
        const float* bp = p.beta + ch0 + cl;
        const bool gb = in_span(gp, 4, p.sp_gamma, p.status) && in_span(bp, 4, p.sp_beta, p.status);
        fold_channel(gb ? __ldg(gp) : 0.0f, gb ? __ldg(bp) : 0.0f, m1, rstd, A, B);
      }
      store16(obase + e * 2, silu_affine<T>(v[b], nk, A, B));
    }
  }
}

// ---------------------------------------------------------------------------
// One-launch group norm + SiLU: x read once.
//
// The N*G spans are cut into chunks of kGnfChunk elements (the last chunk
// of a span may be short); chunk j = span*P + piece.  A persistent CTA per
// SM takes chunks blockIdx.x, blockIdx.x + grid, ... in order, with four
// roles working at once:
//   producer lane: bulk-copies each chunk, and its span's first 16 bytes
//       (K), into a ring of kGnfSlots shared-memory slots;
//   eight stats warps: for each chunk, its sums from shared memory (the
//       same per-thread order and reduction as gn_stats_kernel with
//       kGnfChunk-element pieces), stored as the chunk's tagged record (and
//       K's, for piece 0);
//   kGnfCombiners combiner warps: the CTA's spans in turn (span k to warp
//       k % kGnfCombiners); once this CTA's stats warps have recorded their
//       last chunk of the span (so the other CTAs' records are due too),
//       poll its records and combine them with combine_span into a ring of
//       kGnfCoefSlots coefficient pairs;
//   twelve apply warps: for each chunk, once its span's coefficients are
//       in, silu(x*a + b) from the staged chunk (gamma and beta staged in
//       shared memory when C <= kGnfMaxSmemChannels).
// A slot goes back to the producer when both the stats and the apply warps
// are done with it.  The results equal the two-pass path's with
// kGnfChunk-element pieces bit for bit.
//
// No CTA can wait forever for another: the grid is co-resident (a
// cooperative launch) and a CTA holds at most ceil(P / grid) <= kGnfSlots
// chunks of any span (checked by the host).  Then the lowest unfinished
// span always has all its chunks loaded and recorded: a CTA whose stats
// warps wait for a slot has its apply warps at a chunk kGnfSlots earlier,
// which cannot be in that span.  Every wait is bounded all the same: a wait
// that runs out writes QKNR_ERR_TIMEOUT to *status and sets the
// workspace's abort word to the tag, which the other CTAs' waits watch;
// every warp then leaves its loop, and the producer waits (bounded) for its
// copies in flight before its CTA exits.
//
// In place (out == x) is safe: a chunk is written only after its span's
// records are all in, i.e. after every chunk of the span, the one whose K
// the others copied among them, has been loaded.

constexpr int kGnfStatsWarps = kGnWarps;             // 8: the reduction of gn_stats_kernel
constexpr int kGnfStatsThreads = 32 * kGnfStatsWarps;
constexpr int kGnfApplyWarps = 12;
constexpr int kGnfApplyWarp0 = kGnfStatsWarps;
constexpr int kGnfProducerWarp = kGnfApplyWarp0 + kGnfApplyWarps;
constexpr int kGnfCombiners = 4;
constexpr int kGnfCombinerWarp0 = kGnfProducerWarp + 1;
constexpr int kGnfThreads = 32 * (kGnfCombinerWarp0 + kGnfCombiners);
constexpr int kGnfChunk = 12288;                     // elements per chunk
constexpr int kGnfChunkBytes = kGnfChunk * 2;
constexpr int kGnfStatsVec = kGnfChunk / 8 / kGnfStatsThreads;       // 16-byte vectors per stats thread
constexpr int kGnfApplyVec = kGnfChunk / 8 / (32 * kGnfApplyWarps);   // ... per apply thread
static_assert(kGnfChunk / 8 == kGnfStatsVec * kGnfStatsThreads, "stats warps cover a chunk");
static_assert(kGnfChunk / 8 == kGnfApplyVec * 32 * kGnfApplyWarps, "apply warps cover a chunk");
static_assert(kGnfStatsVec <= kGnBatch, "one batch of gn_stats_kernel covers a chunk (same order)");
constexpr int kGnfSlots = 9;
constexpr int kGnfCoefSlots = 8;
// dynamic shared memory map (bytes)
constexpr int kGnfOffFull = 0;                       // full[kGnfSlots]
constexpr int kGnfOffEmpty = 128;                    // empty[kGnfSlots]
constexpr int kGnfOffCoefFull = 256;                 // coef_full[kGnfCoefSlots]
constexpr int kGnfOffCoefEmpty = 320;                // coef_empty[kGnfCoefSlots]
constexpr int kGnfOffAbort = 384;
constexpr int kGnfOffStatsDone = 388;                // chunks this CTA's stats warps have recorded
constexpr int kGnfOffMeta = 400;                     // [kGnfSlots][2]: first channel, next channel's first element
constexpr int kGnfOffK = 512;                        // [kGnfSlots][16 bytes]: the span's first 16 bytes
constexpr int kGnfOffRed = 768;                      // [2 * kGnWarps] floats
constexpr int kGnfOffCoef = 896;                     // [kGnfCoefSlots][kGnCoefFloats]: m1, rstd, K
constexpr int kGnfOffSlot0 = 1024;
constexpr int kGnfOffGammaBeta = kGnfOffSlot0 + kGnfSlots * kGnfChunkBytes;   // gamma[C], beta[C]
constexpr int kGnfMaxSmemChannels = 1280;            // larger C reads gamma / beta from global memory
constexpr int kGnfSmemBytes = kGnfOffGammaBeta + 8 * kGnfMaxSmemChannels;
constexpr unsigned kGnfFlagStallLoads = 0x1u;        // test: issue no copies
constexpr unsigned kGnfFlagStallRecords = 0x2u;      // test: write no record
static_assert(kGnfOffFull + 8 * kGnfSlots <= kGnfOffEmpty, "shared memory map");
static_assert(kGnfOffEmpty + 8 * kGnfSlots <= kGnfOffCoefFull, "shared memory map");
static_assert(kGnfOffStatsDone + 4 <= kGnfOffMeta, "shared memory map");
static_assert(kGnfOffK + 16 * kGnfSlots <= kGnfOffRed, "shared memory map");
static_assert(kGnfOffMeta + 8 * kGnfSlots <= kGnfOffK, "shared memory map");
static_assert(kGnfOffCoef + 4 * kGnCoefFloats * kGnfCoefSlots <= kGnfOffSlot0, "shared memory map");
static_assert(kGnfSmemBytes <= 227 * 1024, "shared memory map");

struct GnFusedParams {
  const char* x;
  char* out;
  const float* gamma;
  const float* beta;
  unsigned long long* rec;     // [spans][P + 1][2] tagged words
  unsigned* abort_word;        // == tag once a CTA has given up
  int* status;                 // optional
  long long span_len;          // L
  long long hw;                // H * W (a multiple of 8)
  unsigned pieces;             // P = ceil(L / kGnfChunk)
  unsigned total_chunks;       // spans * P
  int groups;
  int group_channels;
  int channels;                // C; gamma and beta are staged in shared memory when <= kGnfMaxSmemChannels
  unsigned tag;                // this call's record tag (nonzero)
  unsigned flags;
  unsigned long long wait_limit_ns;
  float eps;
  // address spans of the buffers (checked builds test every access against them)
  MemSpan sp_x, sp_out, sp_ws, sp_gamma, sp_beta;
};

// (span, piece) of a CTA's chunks blockIdx.x, blockIdx.x + G, ..., kept as
// a running quotient and remainder of the chunk index by P
struct ChunkPos {
  unsigned span, piece;
  __device__ __forceinline__ void init(unsigned j, unsigned P) {
    span = j / P;
    piece = j - span * P;
  }
  __device__ __forceinline__ void advance(unsigned G, unsigned P) {
    piece += G;
    if (piece >= P) {
      const unsigned q = piece / P;
      span += q;
      piece -= q * P;
    }
  }
};

__device__ __forceinline__ void gnf_stats_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGnfStatsThreads) : "memory");
}

struct GnfStatsSync {
  __device__ __forceinline__ void operator()() const { gnf_stats_barrier(); }
};

// bar.sync over the stats warps that also returns whether `pred` held in all
__device__ __forceinline__ bool gnf_stats_barrier_and(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(kGnfStatsThreads)
      : "memory");
  return r != 0;
}

// a wait's first attempt sleeps in the barrier (most complete within it),
// skipping the out-of-line bounded_wait unless it runs out
constexpr uint32_t kGnfSleepNs = 20000;

// one lane's bounded mbarrier wait, its result given to the whole warp
__device__ __forceinline__ bool gnf_warp_wait(uint32_t bar, uint32_t parity, unsigned long long limit,
                                              volatile int* abort_cta, int* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0)
    ok = mbar_try_wait_sleep(bar, parity, kGnfSleepNs) || bounded_wait(bar, parity, limit, abort_cta, status);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// one lane waits (bounded, sleeping) until the shared word reaches `target`;
// the result goes to the whole warp.  Out of line, so it takes the wait
// context as scalars: a struct passed by reference to a call that is not
// inlined would have to live in local memory.
static __device__ __noinline__ bool gnf_wait_local(const volatile unsigned* word, unsigned target, unsigned tag,
                                                   unsigned long long limit_ns, volatile int* abort_cta,
                                                   unsigned* abort_grid, int* status) {
  const RecordWait w{tag, limit_ns, abort_cta, abort_grid, status};
  bool ok = true;
  if ((threadIdx.x & 31) == 0 && *word < target) {
    const unsigned long long t0 = global_timer_ns();
    while (*word < target) {
      if (grid_aborted(w)) {
        ok = false;
        break;
      }
      if (global_timer_ns() - t0 > w.limit_ns) {
        give_up(w);
        ok = false;
        break;
      }
      __nanosleep(256);
    }
  }
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <typename T>
__global__ void __launch_bounds__(kGnfThreads, 1) gn_fused_kernel(const __grid_constant__ GnFusedParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = smem_addr(smem);
  const uint32_t full0 = base + kGnfOffFull;
  const uint32_t empty0 = base + kGnfOffEmpty;
  const uint32_t cfull0 = base + kGnfOffCoefFull;
  const uint32_t cempty0 = base + kGnfOffCoefEmpty;
  volatile int* abort_cta = reinterpret_cast<volatile int*>(smem + kGnfOffAbort);
  volatile unsigned* stats_done = reinterpret_cast<volatile unsigned*>(smem + kGnfOffStatsDone);
  float* coef = reinterpret_cast<float*>(smem + kGnfOffCoef);
  const unsigned G = gridDim.x;
  const unsigned mine = (p.total_chunks - blockIdx.x + G - 1) / G;    // grid <= total_chunks
  const unsigned P = p.pieces;
  const unsigned long long limit = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGnfSlots; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kGnfStatsWarps + kGnfApplyWarps);
    }
    for (int s = 0; s < kGnfCoefSlots; ++s) {
      mbar_init(cfull0 + 8 * s, 1);
      mbar_init(cempty0 + 8 * s, kGnfApplyWarps);
    }
    *abort_cta = 0;
    *stats_done = 0;
    fence_barrier_init();
  }
  const bool gb_smem = p.channels <= kGnfMaxSmemChannels;
  float* sgamma = reinterpret_cast<float*>(smem + kGnfOffGammaBeta);
  float* sbeta = sgamma + kGnfMaxSmemChannels;
  if (gb_smem) {
    for (int c = threadIdx.x; c < p.channels; c += blockDim.x) {
      const bool gb = in_span(p.gamma + c, 4, p.sp_gamma, p.status) && in_span(p.beta + c, 4, p.sp_beta, p.status);
      sgamma[c] = gb ? __ldg(p.gamma + c) : 0.0f;
      sbeta[c] = gb ? __ldg(p.beta + c) : 0.0f;
    }
  }
  __syncthreads();

  ChunkPos pos;
  pos.init(blockIdx.x, P);

  if (warp == kGnfProducerWarp) {
    // ---------------- producer: one lane; per chunk a bulk copy of the chunk
    // and one of its span's first 16 bytes, both counted on the slot's barrier
    if (lane != 0) return;
    unsigned issued = 0;
    bool ok = true;
    int s = 0;
    uint32_t ph = 0;
    for (unsigned t = 0; t < mine; ++t, pos.advance(G, P)) {
      const uint32_t empty = empty0 + 8 * s;
      if (!mbar_try_wait_sleep(empty, ph ^ 1u, kGnfSleepNs) &&
          !bounded_wait(empty, ph ^ 1u, limit, abort_cta, p.status)) {
        ok = false;
        break;
      }
      if (*abort_cta) {
        ok = false;
        break;
      }
      if (p.flags & kGnfFlagStallLoads) break;
      const long long lo = static_cast<long long>(pos.piece) * kGnfChunk;
      const long long rest = p.span_len - lo;
      const uint32_t bytes = static_cast<uint32_t>(rest < kGnfChunk ? rest : kGnfChunk) * 2u;
      const uint32_t full = full0 + 8 * s;
      const char* span_x = p.x + static_cast<long long>(pos.span) * p.span_len * 2;
      // the chunk's first channel (within the group) and where the next one
      // starts, for the apply warps; published by the arrive below
      const unsigned cl = channel_of(lo, p.hw);
      unsigned* meta = reinterpret_cast<unsigned*>(smem + kGnfOffMeta + 8 * s);
      meta[0] = cl;
      meta[1] = (cl + 1u) * static_cast<unsigned>(p.hw);
      // checked builds: the chunk and the span's first 16 bytes inside x
      // (the slot map is fixed at compile time), else nothing more is issued
      if (!in_span(span_x + lo * 2, bytes, p.sp_x, p.status) || !in_span(span_x, 16u, p.sp_x, p.status)) {
        give_up(RecordWait{p.tag, limit, abort_cta, p.abort_word, p.status});
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(full, bytes + 16u);
      bulk_load(base + kGnfOffSlot0 + s * kGnfChunkBytes, span_x + lo * 2, bytes, full);
      bulk_load(base + kGnfOffK + 16 * s, span_x, 16u, full);
      ++issued;
      if (++s == kGnfSlots) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (!ok || *abort_cta) {
      // wait (bounded) for the copies of the latest use of every slot
      const unsigned first = issued > kGnfSlots ? issued - kGnfSlots : 0;
      for (unsigned it = first; it < issued; ++it) {
        const uint32_t bar = full0 + 8 * (it % kGnfSlots);
        const uint32_t phase = (it / kGnfSlots) & 1u;
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(bar, phase) && global_timer_ns() - t0 < limit) {
        }
      }
    }
    return;
  }

  if (warp >= kGnfCombinerWarp0) {
    // ---------------- combiners: the coefficients of the CTA's spans
    const int c = warp - kGnfCombinerWarp0;
    const RecordWait rw{p.tag, limit, abort_cta, p.abort_word, p.status};
    unsigned k = 0;                                  // the CTA's k-th span
    for (unsigned t = 0; t < mine;) {
      // this CTA's chunks of the span: t .. t_end - 1
      const unsigned span = pos.span;
      unsigned t_end = t;
      while (t_end < mine && pos.span == span) {
        ++t_end;
        pos.advance(G, P);
      }
      t = t_end;
      const unsigned kk = k++;
      if (kk % kGnfCombiners != static_cast<unsigned>(c)) continue;
      const int e = static_cast<int>(kk % kGnfCoefSlots);
      const uint32_t use_parity = (kk / kGnfCoefSlots) & 1u;
      if (!gnf_warp_wait(cempty0 + 8 * e, use_parity ^ 1u, limit, abort_cta, p.status)) break;
      if (!gnf_wait_local(stats_done, t_end, rw.tag, rw.limit_ns, rw.abort_cta, rw.abort_grid, rw.status)) break;
      if (!combine_span<true>(p.rec + static_cast<long long>(span) * (P + 1) * 2, static_cast<int>(P), p.span_len,
                              kGnfChunk, p.eps, &rw, coef + kGnCoefFloats * e, p.sp_ws, p.status)) {
        if (kChecked) give_up(rw);                   // a record range outside the workspace
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(cfull0 + 8 * e);    // release: the coefficients are visible
    }
    return;
  }

  if (warp >= kGnfApplyWarp0) {
    // ---------------- apply warps: each on its own, no barrier among them
    const int at = (warp - kGnfApplyWarp0) * 32 + lane;
    unsigned cached_span = 0xffffffffu;
    unsigned nspans = 0;
    int ch0 = 0;
    float m1 = 0.0f, rstd = 0.0f;
    float2 nk = make_float2(0.0f, 0.0f);
    int s = 0;
    uint32_t ph = 0;
    for (unsigned u = 0; u < mine; ++u, pos.advance(G, P)) {
      const unsigned span = pos.span;
      if (span != cached_span) {
        // hand back the previous span's coefficients (held in registers),
        // then take this span's
        if (nspans > 0) {
          __syncwarp();
          if (lane == 0) mbar_arrive(cempty0 + 8 * ((nspans - 1) % kGnfCoefSlots));
        }
        const int e = static_cast<int>(nspans % kGnfCoefSlots);
        if (!gnf_warp_wait(cfull0 + 8 * e, (nspans / kGnfCoefSlots) & 1u, limit, abort_cta, p.status)) break;
        m1 = coef[kGnCoefFloats * e];
        rstd = coef[kGnCoefFloats * e + 1];
        nk = make_float2(-coef[kGnCoefFloats * e + 2], -coef[kGnCoefFloats * e + 2]);
        ch0 = static_cast<int>(span % static_cast<unsigned>(p.groups)) * p.group_channels;
        cached_span = span;
        ++nspans;
      }
      if (!gnf_warp_wait(full0 + 8 * s, ph, limit, abort_cta, p.status)) break;
      const unsigned lo = pos.piece * static_cast<unsigned>(kGnfChunk);     // < L < 2^31
      const unsigned rest = static_cast<unsigned>(p.span_len) - lo;
      const int nvec = static_cast<int>(rest < kGnfChunk ? rest : kGnfChunk) / 8;
      char* obase = p.out + (static_cast<long long>(span) * p.span_len + lo) * 2;
      // checked builds: the chunk's output inside out, else it is not written
      const bool out_ok = in_span(obase, static_cast<unsigned long long>(nvec) * 16, p.sp_out, p.status);
      const unsigned char* slot = smem + kGnfOffSlot0 + s * kGnfChunkBytes;
      const unsigned hw = static_cast<unsigned>(p.hw);
      const uint2 meta = *reinterpret_cast<const uint2*>(smem + kGnfOffMeta + 8 * s);
      unsigned ch_end = meta.y;
      // gamma and beta of channel ch (checked builds: inside the staged
      // copies or the buffers)
      auto fold = [&](int ch, float2& A_, float2& B_) {
        bool ok;
        if (gb_smem) {
          ok = !kChecked || (ch >= 0 && ch < p.channels);
          if (!ok && p.status) atomicCAS(p.status, 0, kStatusBounds);
        } else {
          ok = in_span(p.gamma + ch, 4, p.sp_gamma, p.status) && in_span(p.beta + ch, 4, p.sp_beta, p.status);
        }
        const float g = ok ? (gb_smem ? sgamma[ch] : __ldg(p.gamma + ch)) : 0.0f;
        const float be = ok ? (gb_smem ? sbeta[ch] : __ldg(p.beta + ch)) : 0.0f;
        fold_channel(g, be, m1, rstd, A_, B_);
      };
      float2 A, B;
      fold(ch0 + static_cast<int>(meta.x), A, B);
      auto one = [&](int v) {
        const uint4 raw = *reinterpret_cast<const uint4*>(slot + v * 16);
        const unsigned e = lo + static_cast<unsigned>(v) * 8u;
        if (e >= ch_end) {
          const unsigned cl = e / hw;
          ch_end = (cl + 1u) * hw;
          fold(ch0 + static_cast<int>(cl), A, B);
        }
        if (out_ok) store16(obase + v * 16, silu_affine<T>(raw, nk, A, B));
      };
      if (nvec == kGnfChunk / 8) {
#pragma unroll
        for (int b = 0; b < kGnfApplyVec; ++b) one(at + b * 32 * kGnfApplyWarps);
      } else {
#pragma unroll
        for (int b = 0; b < kGnfApplyVec; ++b)
          if (at + b * 32 * kGnfApplyWarps < nvec) one(at + b * 32 * kGnfApplyWarps);
      }
      // the slot has been read for the last time by this warp
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
      if (++s == kGnfSlots) {
        s = 0;
        ph ^= 1u;
      }
    }
    return;
  }

  // ---------------- stats warps
  const int tid = threadIdx.x;                       // 0 .. kGnfStatsThreads - 1
  float* red = reinterpret_cast<float*>(smem + kGnfOffRed);
  int s = 0;
  uint32_t ph = 0;
  for (unsigned t = 0; t < mine; ++t, pos.advance(G, P)) {
    const bool got = mbar_try_wait_sleep(full0 + 8 * s, ph, kGnfSleepNs) ||
                     bounded_wait(full0 + 8 * s, ph, limit, abort_cta, p.status);
    if (!gnf_stats_barrier_and(got)) {
      if (tid == 0) atomicExch(p.abort_word, p.tag);
      break;                                         // every stats warp leaves together
    }
    const unsigned span = pos.span, piece = pos.piece;
    const long long lo = static_cast<long long>(piece) * kGnfChunk;
    const long long rest = p.span_len - lo;
    const int nvec = static_cast<int>(rest < kGnfChunk ? rest : kGnfChunk) / 8;
    float2 first[4];
    Elem<T>::unpack(*reinterpret_cast<const uint4*>(smem + kGnfOffK + 16 * s), first);
    const float K = shift_of_first8(first);
    const unsigned char* slot = smem + kGnfOffSlot0 + s * kGnfChunkBytes;
    // vectors tid, tid + kGnfStatsThreads, ... of the chunk, summed around
    // the first value of the first one (as gn_stats_kernel)
    const int my_vec = tid < nvec ? (nvec - 1 - tid) / kGnfStatsThreads + 1 : 0;
    float kt = 0.0f;
    if (my_vec > 0) {
      float2 f[4];
      Elem<T>::unpack(*reinterpret_cast<const uint4*>(slot + tid * 16), f);
      kt = f[0].x;
    }
    const float2 nk = make_float2(-kt, -kt);
    float2 a1 = make_float2(0.0f, 0.0f), a2 = make_float2(0.0f, 0.0f);
    auto one = [&](int v) {
      float2 X[4];
      Elem<T>::unpack(*reinterpret_cast<const uint4*>(slot + v * 16), X);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 d = __fadd2_rn(X[q], nk);
        a1 = __fadd2_rn(a1, d);
        a2 = __ffma2_rn(d, d, a2);
      }
    };
    if (nvec == kGnfChunk / 8) {
#pragma unroll
      for (int b = 0; b < kGnfStatsVec; ++b) one(tid + b * kGnfStatsThreads);
    } else {
#pragma unroll
      for (int b = 0; b < kGnfStatsVec; ++b)
        if (tid + b * kGnfStatsThreads < nvec) one(tid + b * kGnfStatsThreads);
    }
    // this warp has read the slot for the last time
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    const Moments pm = piece_moments(
        moments_of(8.0f * static_cast<float>(my_vec), __fsub_rn(kt, K), __fadd_rn(a1.x, a1.y), __fadd_rn(a2.x, a2.y)),
        nvec, red, GnfStatsSync());
    if (tid == 0) {
      if (!(p.flags & kGnfFlagStallRecords)) {
        unsigned long long* rec = p.rec + static_cast<long long>(span) * (P + 1) * 2;
        st_record(rec + 2 * piece, tagged(p.tag, pm.u), tagged(p.tag, pm.m));
        if (piece == 0) st_record(rec + 2 * P, tagged(p.tag, K), tagged(p.tag, 0.0f));
      }
      *stats_done = t + 1;
    }
    // red[] is rewritten by the next chunk only after every stats warp has
    // passed that chunk's first barrier, which thread 0 reaches after
    // reading it here
    if (++s == kGnfSlots) {
      s = 0;
      ph ^= 1u;
    }
  }
}

}  // namespace qknr
