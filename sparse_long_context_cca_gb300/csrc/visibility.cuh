// The visible set of a query row, as every kernel of this library applies it
// ("Core Context Aware Transformers for Long Context Language Modeling", Method
// section, fusion equation; 0-indexed).  Query i sees
//   - the raw tokens of its window, from window_start(i) to i, where the window
//     begins at window_lo(i) = max(0, i - w + 1), or, with window_mode 1, at the
//     group boundary g * (window_lo(i) / g) so that no token falls in a gap;
//   - the core tokens j < visible_cores(i) = window_lo(i) / g, i.e. the groups
//     that lie wholly before window_lo(i).
#pragma once

namespace cca {

__host__ __device__ __forceinline__ int window_lo(int i, int w) { return i - w + 1 > 0 ? i - w + 1 : 0; }
__host__ __device__ __forceinline__ int visible_cores(int i, int w, int g) { return window_lo(i, w) / g; }
__host__ __device__ __forceinline__ int window_start(int i, int w, int g, int window_mode) {
    const int lo = window_lo(i, w);
    return window_mode ? (lo / g) * g : lo;
}

}  // namespace cca
