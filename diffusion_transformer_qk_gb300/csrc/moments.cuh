// Mean and variance of many values in fp32, robust to a reference value
// that lies far from the mean (the AdaLN and group-norm statistics).
//
// A part of the values is (n, u, m): its count n, its mean u taken
// relative to a reference R common to every part, and m, the sum of
// squared deviations from its own mean.  A thread forms its part (or one
// per batch of its values) from sums around its own first value k, s1 =
// sum (x - k) and s2 = sum (x - k)^2, so the cancellation in m = s2 - s1^2
// / n is bounded by those few values.  Parts are merged around the mean r of one of them (the
// pairwise-update identity of Chan, Golub and LeVeque, "Updating formulae
// and a pairwise algorithm for computing sample variances", 1979, summed
// over all parts at once):
//
//     a = sum n_i (u_i - r),   c = sum (m_i + n_i (u_i - r)^2),
//     N = sum n_i,  u = r + a / N,  m = c - a^2 / N,
//
// so every level of a reduction is plain sums of independent terms, and
// the one cancellation left, in c - a^2 / N, is bounded by how far the
// reference part's mean lies from the merged mean.  Sums of (x - R)^2
// around a single value R instead lose the variance to cancellation once R
// is far from the mean against the spread (a first element that is an
// outlier).
#pragma once

namespace qknr {

struct Moments {
  float n;   // count
  float u;   // mean - R
  float m;   // sum of squared deviations from the mean
};

// 1/x on the special-function unit (rcp.approx, about 1 ulp)
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The part of n values whose sums around k are s1 and s2; k_minus_r = k - R.
__device__ __forceinline__ Moments moments_of(float n, float k_minus_r, float s1, float s2) {
  Moments r{n, 0.0f, 0.0f};
  if (n > 0.0f) {
    const float mean = __fmul_rn(s1, rcp_approx(n));        // mean of x - k
    r.u = __fadd_rn(k_minus_r, mean);
    r.m = fmaxf(__fmaf_rn(-s1, mean, s2), 0.0f);             // s2 - s1^2 / n
  }
  return r;
}

// Running sums a and c of parts around the reference mean r.
struct RefSums {
  float a = 0.0f, c = 0.0f;
  __device__ __forceinline__ void add(const Moments& p, float r) {
    const float d = __fsub_rn(p.u, r);
    const float nd = __fmul_rn(p.n, d);
    a = __fadd_rn(a, nd);
    c = __fadd_rn(c, __fmaf_rn(nd, d, p.m));
  }
};

// The merged part of parts with N values in all, from their sums around r.
__device__ __forceinline__ Moments merged(float n, float r, const RefSums& s) {
  Moments o{n, 0.0f, 0.0f};
  if (n > 0.0f) {
    const float da = __fmul_rn(s.a, rcp_approx(n));
    o.u = __fadd_rn(r, da);
    o.m = fmaxf(__fmaf_rn(-s.a, da, s.c), 0.0f);
  }
  return o;
}

// The merged part of a warp's lanes (n_warp values in all; lanes with no
// values pass n = 0), around lane 0's mean: an xor tree of plain sums, the
// same result in every lane.  Lane 0 holds values whenever any lane does.
__device__ __forceinline__ Moments warp_moments(const Moments& v, float n_warp) {
  const float r = __shfl_sync(0xffffffffu, v.u, 0);
  RefSums s;
  s.add(v, r);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    s.a = __fadd_rn(s.a, __shfl_xor_sync(0xffffffffu, s.a, off));
    s.c = __fadd_rn(s.c, __shfl_xor_sync(0xffffffffu, s.c, off));
  }
  return merged(n_warp, r, s);
}

// The shift of a row's or group's statistics and output: the lower median
// (4th smallest) of its first 8 values v.  It is one of the values, so x - K
// is exact for values near it, and it lies among the bulk unless 4 of the 8
// are outliers, which keeps mean - K small and exactly representable to
// fp32 precision of its own size.  A sorting network of 19 compare-swaps.
__device__ __forceinline__ float shift_of_first8(const float2 (&v)[4]) {
  float a[8] = {v[0].x, v[0].y, v[1].x, v[1].y, v[2].x, v[2].y, v[3].x, v[3].y};
  constexpr int kNet[19][2] = {{0, 2}, {1, 3}, {4, 6}, {5, 7}, {0, 4}, {1, 5}, {2, 6}, {3, 7}, {0, 1},
                               {2, 3}, {4, 5}, {6, 7}, {2, 4}, {3, 5}, {1, 4}, {3, 6}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
  for (int i = 0; i < 19; ++i) {
    const float lo = fminf(a[kNet[i][0]], a[kNet[i][1]]), hi = fmaxf(a[kNet[i][0]], a[kNet[i][1]]);
    a[kNet[i][0]] = lo;
    a[kNet[i][1]] = hi;
  }
  return a[3];
}

// Values a warp covers when T threads take items j, j + T, j + 2T, ... of
// V items of `per` values each: 32 * (V / T) items plus the warp's share of
// the V % T left over, lanes 32w .. 32w + 31.
__device__ __forceinline__ float warp_count(int w, int V, int T, int per) {
  const int q = V / T, r = V - (V / T) * T;
  int extra = r - 32 * w;
  extra = extra < 0 ? 0 : (extra > 32 ? 32 : extra);
  return static_cast<float>((32 * q + extra) * per);
}

}  // namespace qknr
