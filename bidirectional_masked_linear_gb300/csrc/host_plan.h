// host_plan.h -- host-side planning of lion_attn_fwd_host (plain C++, no
// CUDA): how the batch is cut into slices.
#pragma once

namespace lion {

// Batch rows [bounds[s], bounds[s + 1]) of slice s: with S >= 3 (and enough
// rows) the first and last slices weigh 1/2 and the others 1; returns the
// number of slices.
constexpr int kMaxSlices = 64;
inline int slice_bounds(int B, int S, int* bounds) {
  if (S < 1) S = 1;
  if (S > B) S = B;
  const bool taper = S >= 3 && B >= 2 * S;
  const double total = taper ? S - 1.0 : (double)S;
  double acc = 0.0;
  bounds[0] = 0;
  for (int s = 0; s < S; ++s) {
    acc += taper && (s == 0 || s == S - 1) ? 0.5 : 1.0;
    int b = (int)(acc / total * B + 0.5);
    if (b <= bounds[s]) b = bounds[s] + 1;          // every slice holds a row
    if (b > B - (S - 1 - s)) b = B - (S - 1 - s);   // and leaves one for each slice after it
    bounds[s + 1] = b;
  }
  bounds[S] = B;
  return S;
}

}  // namespace lion
