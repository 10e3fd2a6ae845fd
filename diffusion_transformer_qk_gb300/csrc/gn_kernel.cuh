// Group norm + SiLU kernels for sm_103a ("fused qknorm rope Flux 2.0",
// section "Not in this PR — follow-ups": group_norm_silu for the VAE).
//
// Activations are NCHW, so the (C/G)*H*W elements of sample n, group g are
// one contiguous span.  A group has few and large spans (32 groups of up to
// millions of elements in a VAE decoder), so each span is cut into P pieces
// and the work runs in two stream-ordered launches, with no CTA ever
// waiting for another:
//
//   stats: one CTA per piece; 16-byte loads; per-thread fp32 sums of
//          (x - K) and (x - K)^2 around the span's first element K, then an
//          fp64 reduction over the CTA into workspace[span][piece] = (S1, S2);
//          piece 0 also records K in workspace[span][P].
//   apply: one CTA per piece; it adds its span's P partials in fixed order
//          (fp64), forms mean = K + S1/L and var = S2/L - (S1/L)^2, folds
//          a = gamma[c]/sqrt(var + eps), b = beta[c] - mean*a per channel,
//          and writes silu(x*a + b) = y / (1 + exp(-y)).
//
// The host issues the pair once for all groups, or per batch of groups
// (a batch small enough for L2 lets the apply launch re-read from L2).
#pragma once

#include "qknr_ptx.cuh"

namespace qknr {

constexpr int kGnThreads = 256;
constexpr int kGnBatch = 8;          // 16-byte loads a thread keeps in flight

struct GnParams {
  const char* x;
  char* out;
  const float* gamma;
  const float* beta;
  double* partial;             // [spans][pieces + 1][2]: S1, S2 of each piece; then (K, 0)
  long long span_len;          // L = (C/G) * H * W elements
  long long hw;                // H * W (a multiple of 8)
  long long piece_len;         // elements per piece (a multiple of 8)
  int channels;                // C
  int groups;                  // G
  int group_channels;          // C / G
  int pieces;                  // P pieces per span
  int span0;                   // first span (n*G + g) of this launch
  float eps;
};

// sum of a double over the CTA (kGnThreads threads); valid in thread 0
__device__ __forceinline__ double cta_sum(double v, double* red) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < kGnThreads / 32; ++w) t += red[w];
  __syncthreads();
  return t;
}

template <typename T>
__global__ void __launch_bounds__(kGnThreads) gn_stats_kernel(const __grid_constant__ GnParams p) {
  __shared__ double red[2][kGnThreads / 32];
  const int span = p.span0 + blockIdx.y;
  const int piece = blockIdx.x;
  const char* base = p.x + static_cast<long long>(span) * p.span_len * 2;
  const long long lo = static_cast<long long>(piece) * p.piece_len;
  long long hi = lo + p.piece_len;
  if (hi > p.span_len) hi = p.span_len;
  float2 first[4];
  Elem<T>::unpack(__ldg(reinterpret_cast<const uint4*>(base)), first);
  const float2 nk = make_float2(-first[0].x, -first[0].x);
  float2 a1 = make_float2(0.0f, 0.0f), a2 = make_float2(0.0f, 0.0f);
  // kGnBatch independent 16-byte loads in flight per thread before any is used
  constexpr long long kStride = kGnThreads * 8;
  for (long long e0 = lo + threadIdx.x * 8; e0 < hi; e0 += kStride * kGnBatch) {
    uint4 v[kGnBatch];
#pragma unroll
    for (int b = 0; b < kGnBatch; ++b) {
      const long long e = e0 + b * kStride;
      v[b] = e < hi ? __ldg(reinterpret_cast<const uint4*>(base + e * 2)) : make_uint4(0, 0, 0, 0);
    }
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
      }
    }
  }
  const double s1 = cta_sum(static_cast<double>(a1.x) + static_cast<double>(a1.y), red[0]);
  const double s2 = cta_sum(static_cast<double>(a2.x) + static_cast<double>(a2.y), red[1]);
  if (threadIdx.x == 0) {
    double* rec = p.partial + static_cast<long long>(span) * (p.pieces + 1) * 2;
    rec[2 * piece] = s1;
    rec[2 * piece + 1] = s2;
    if (piece == 0) {
      // the shift, kept here because an in-place apply overwrites x
      rec[2 * p.pieces] = static_cast<double>(first[0].x);
      rec[2 * p.pieces + 1] = 0.0;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kGnThreads) gn_apply_kernel(const __grid_constant__ GnParams p) {
  __shared__ float coef[2];                  // mean and 1/sqrt(var + eps) of the span
  const int span = p.span0 + blockIdx.y;
  const int piece = blockIdx.x;
  const char* base = p.x + static_cast<long long>(span) * p.span_len * 2;
  char* obase = p.out + static_cast<long long>(span) * p.span_len * 2;
  if (threadIdx.x == 0) {
    const double* rec = p.partial + static_cast<long long>(span) * (p.pieces + 1) * 2;
    double s1 = 0.0, s2 = 0.0;
    for (int i = 0; i < p.pieces; ++i) {
      s1 += rec[2 * i];
      s2 += rec[2 * i + 1];
    }
    const double inv_l = 1.0 / static_cast<double>(p.span_len);
    const double m1 = s1 * inv_l;
    double var = s2 * inv_l - m1 * m1;
    var = var > 0.0 ? var : 0.0;
    coef[0] = static_cast<float>(rec[2 * p.pieces] + m1);
    coef[1] = static_cast<float>(1.0 / sqrt(var + static_cast<double>(p.eps)));
  }
  __syncthreads();
  const float mean = coef[0], rstd = coef[1];
  const int g = span % p.groups;
  const long long lo = static_cast<long long>(piece) * p.piece_len;
  long long hi = lo + p.piece_len;
  if (hi > p.span_len) hi = p.span_len;
  // channel of the current chunk (a 16-byte chunk never straddles a
  // channel: H*W is a multiple of 8), refreshed only when a chunk crosses
  // into the next channel, with its folded coefficients a and b
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
        const long long cl = e / p.hw;
        ch_end = (cl + 1) * p.hw;
        const int c = g * p.group_channels + static_cast<int>(cl);
        const float a = __fmul_rn(__ldg(p.gamma + c), rstd);
        const float bb = __fmaf_rn(-mean, a, __ldg(p.beta + c));
        A = make_float2(a, a);
        B = make_float2(bb, bb);
      }
      float2 X[4], O[4];
      Elem<T>::unpack(v[b], X);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 y = __ffma2_rn(X[j], A, B);
        O[j] = make_float2(__fdividef(y.x, 1.0f + __expf(-y.x)), __fdividef(y.y, 1.0f + __expf(-y.y)));
      }
      store16(obase + e * 2, Elem<T>::pack(O));
    }
  }
}

}  // namespace qknr
